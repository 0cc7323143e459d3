"""Seeded synthetic inputs shared by the tests, the bench and the oracle checks.

This module holds no arithmetic of the scoring method: it only draws paged K
caches, block vectors and anchors with planted topics. Every random value is
a pure function of (seed, stream, element counter) through SplitMix64
(Steele, Lea & Flood, "Fast splittable pseudorandom number generators",
OOPSLA 2014). Noise is the Irwin-Hall sum of twelve 16-bit uniforms minus 6
(mean 0, variance 1 up to 2^-32), formed in integer arithmetic and scaled by
2^-17, so the float32 value is exact. A Key element is

    K = fl32(cs[topic][d] + fl32(sigma[l,h] * noise))

with both operations rounded to nearest (no fused multiply-add), and stored
as float32 or as bf16 by round-to-nearest-even of those float32 bits. The
numpy generator here and the CUDA generator in ``synth/csrc/synth.cu`` are
two implementations of that one definition and agree bit for bit.
"""
from __future__ import annotations

import ctypes
import dataclasses
import os
from typing import Optional

import numpy as np

GOLDEN = 0x9E3779B97F4A7C15
M1 = 0xBF58476D1CE4E5B9
M2 = 0x94D049BB133111EB
MASK64 = (1 << 64) - 1
F32_NAN_BITS = 0x7FC00000
BF16_NAN_BITS = 0x7FC0


def _mix64_int(z: int) -> int:
    z &= MASK64
    z = ((z ^ (z >> 30)) * M1) & MASK64
    z = ((z ^ (z >> 27)) * M2) & MASK64
    return z ^ (z >> 31)


def stream_key(seed: int, stream: int) -> int:
    """64-bit key of one random stream (one per kind of table) of a seed."""
    return _mix64_int((seed * GOLDEN + stream * 0xD1B54A32D192ED03) & MASK64)


def mix64(z: np.ndarray) -> np.ndarray:
    """SplitMix64 output function on a uint64 array (wrapping arithmetic)."""
    z = z.astype(np.uint64, copy=True)
    with np.errstate(over="ignore"):
        z ^= z >> np.uint64(30)
        z *= np.uint64(M1)
        z ^= z >> np.uint64(27)
        z *= np.uint64(M2)
        z ^= z >> np.uint64(31)
    return z


def noise(key: int, counters: np.ndarray) -> np.ndarray:
    """float32 noise for each uint64 element counter (see module docstring)."""
    c = counters.astype(np.uint64)
    total = np.zeros(c.shape, dtype=np.int64)
    with np.errstate(over="ignore"):
        for k in range(3):
            h = mix64(np.uint64(key) + (np.uint64(3) * c + np.uint64(k + 1)) * np.uint64(GOLDEN))
            for sh in (0, 16, 32, 48):
                total += ((h >> np.uint64(sh)) & np.uint64(0xFFFF)).astype(np.int64)
    num = 2 * total + 12 - 786432
    return num.astype(np.float32) * np.float32(2.0**-17)


def bf16_rne(x: np.ndarray) -> np.ndarray:
    """float32 -> bf16 bits, round to nearest even (finite inputs)."""
    u = np.asarray(x, dtype=np.float32).view(np.uint32).astype(np.uint64)
    r = ((u >> np.uint64(16)) & np.uint64(1)) + np.uint64(0x7FFF)
    return ((u + r) >> np.uint64(16)).astype(np.uint16)


def element_f32(cs_row: np.ndarray, sigma: np.ndarray, nz: np.ndarray) -> np.ndarray:
    """fl32(cs + fl32(sigma * noise)), element-wise, in float32."""
    prod = (np.asarray(sigma, dtype=np.float32) * nz).astype(np.float32)
    return (np.asarray(cs_row, dtype=np.float32) + prod).astype(np.float32)


# --------------------------------------------------------------------------
# workload specifications
# --------------------------------------------------------------------------


@dataclasses.dataclass
class CacheSpec:
    """A paged K cache with planted topics, its block table and step sizes."""

    name: str
    L: int
    H: int
    D: int
    bs: int
    dtype: str  # "f32" or "bf16"
    seq_lens: list
    num_topics: int
    scale: float
    W: int
    K: int
    seed: int
    sigma_range: Optional[tuple] = None  # per-(layer, head) sigma ~ U[a, b]; None -> 1
    weighted: bool = False
    shuffle_pages: bool = False
    span: int = 0  # tokens per topic segment; 0 -> bs
    extra_pages: int = 0  # unused physical pages in the pool
    layout: str = "LPHTD"  # or "LPTHD" (token-major inside a page), "PLHTD" (page-major)

    # ---- derived -------------------------------------------------------
    def __post_init__(self):
        self.seq_lens = [int(t) for t in self.seq_lens]
        if self.span == 0:
            self.span = self.bs
        assert self.span % self.bs == 0
        nb = [(t + self.bs - 1) // self.bs for t in self.seq_lens]
        self.nb = nb
        self.offsets = np.concatenate([[0], np.cumsum(nb)]).astype(np.int32)
        self.total_blocks = int(self.offsets[-1])
        self.num_pages = self.total_blocks + self.extra_pages
        rng = np.random.default_rng(self.seed)
        # centroids: normalised N(0, I_D) directions, scaled (float64 -> float32)
        c = rng.standard_normal((self.num_topics, self.D))
        c /= np.linalg.norm(c, axis=1, keepdims=True)
        self.centroids = c
        self.cs = (self.scale * c).astype(np.float32)
        if self.sigma_range is None:
            self.sigma = np.ones((self.L, self.H), dtype=np.float32)
        else:
            a, b = self.sigma_range
            self.sigma = rng.uniform(a, b, size=(self.L, self.H)).astype(np.float32)
        # topics per segment, balanced counts per request, shuffled; the
        # request's query topic is the topic of its last segment
        topics, q = [], []
        for t in self.seq_lens:
            nseg = max(1, (t + self.span - 1) // self.span)
            seg = rng.permutation(np.arange(nseg) % self.num_topics)
            topics.append(seg)
            q.append(int(seg[-1]))
        self.segment_topics = topics
        self.query_topic = np.array(q, dtype=np.int32)
        bpseg = self.span // self.bs
        self.block_topic = np.concatenate(
            [np.repeat(seg, bpseg)[:n] for seg, n in zip(topics, nb)]
        ).astype(np.int32) if self.total_blocks else np.zeros(0, np.int32)
        # physical page of each logical block
        if self.shuffle_pages:
            self.pages = rng.permutation(self.num_pages)[: self.total_blocks].astype(np.int32)
        else:
            self.pages = np.arange(self.total_blocks, dtype=np.int32)
        nv = []
        for t, n in zip(self.seq_lens, nb):
            for j in range(n):
                nv.append(min(self.bs, t - j * self.bs))
        self.n_valid = np.array(nv, dtype=np.int32)
        tok0 = []
        base = 0
        for t, n in zip(self.seq_lens, nb):
            for j in range(n):
                tok0.append(base + j * self.bs)
            base += t
        self.block_tok0 = np.array(tok0, dtype=np.int64)
        self.key = stream_key(self.seed, 1)

    @property
    def R(self) -> int:
        return len(self.seq_lens)

    @property
    def elem_bytes(self) -> int:
        return 4 if self.dtype == "f32" else 2

    @property
    def shape(self):
        """Logical [L][P][H][bs][D] shape of the paged cache."""
        return (self.L, self.num_pages, self.H, self.bs, self.D)

    def strides(self):
        """Element strides (layer, page, head, token); the dim stride is 1."""
        L, P, H, bs, D = self.shape
        if self.layout == "LPHTD":
            return (P * H * bs * D, H * bs * D, bs * D, D)
        if self.layout == "LPTHD":
            return (P * bs * H * D, bs * H * D, D, H * D)
        if self.layout == "PLHTD":
            return (H * bs * D, L * H * bs * D, bs * D, D)
        raise ValueError(self.layout)

    def storage_elems(self) -> int:
        L, P, H, bs, D = self.shape
        return L * P * H * bs * D

    def k_bytes(self) -> int:
        """Bytes of valid Keys (the pool's algorithmic read volume)."""
        return int(sum(self.seq_lens)) * self.L * self.H * self.D * self.elem_bytes

    def pages_of(self, r: int) -> np.ndarray:
        return self.pages[self.offsets[r] : self.offsets[r + 1]]


def view_paged(storage: np.ndarray, spec: CacheSpec) -> np.ndarray:
    """[L][P][H][bs][D] view of a flat storage array laid out as ``spec``."""
    es = storage.dtype.itemsize
    st = tuple(s * es for s in spec.strides()) + (es,)
    return np.lib.stride_tricks.as_strided(storage, shape=spec.shape, strides=st)


def gen_paged_numpy(spec: CacheSpec) -> np.ndarray:
    """Flat storage (float32 or bf16 bits) of the paged cache, on the host.

    Positions past a block's valid tokens, and unused pages, hold NaN.
    Meant for small caches (tests); the CUDA generator makes large ones.
    """
    dt = np.float32 if spec.dtype == "f32" else np.uint16
    storage = np.empty(spec.storage_elems(), dtype=dt)
    storage.view(np.uint32 if dt == np.float32 else np.uint16)[:] = (
        F32_NAN_BITS if dt == np.float32 else BF16_NAN_BITS
    )
    kc = view_paged(storage, spec)
    L, H, D, bs = spec.L, spec.H, spec.D, spec.bs
    l_ix, h_ix, t_ix, d_ix = np.meshgrid(
        np.arange(L), np.arange(H), np.arange(bs), np.arange(D), indexing="ij"
    )
    for g in range(spec.total_blocks):
        n = int(spec.n_valid[g])
        tok = spec.block_tok0[g] + t_ix[:, :, :n, :]
        ctr = (((tok * L + l_ix[:, :, :n, :]) * H + h_ix[:, :, :n, :]) * D + d_ix[:, :, :n, :]).astype(np.uint64)
        nz = noise(spec.key, ctr)
        sig = spec.sigma[l_ix[:, :, :n, :], h_ix[:, :, :n, :]]
        cs = spec.cs[spec.block_topic[g]][d_ix[:, :, :n, :]]
        v = element_f32(cs, sig, nz)  # [L][H][n][D]
        blk = v if spec.dtype == "f32" else bf16_rne(v)
        kc[:, int(spec.pages[g]), :, :n, :] = blk
    return storage


@dataclasses.dataclass
class RowsSpec:
    """N rows of D values: fl32(cs[topic] + sigma * noise), topics balanced and shuffled."""

    N: int
    D: int
    num_topics: int
    scale: float
    sigma: float
    seed: int
    stream: int
    dtype: str = "f32"
    topics: Optional[np.ndarray] = None
    centroid_seed: Optional[int] = None  # share centroids with another spec

    def __post_init__(self):
        rng = np.random.default_rng(self.centroid_seed if self.centroid_seed is not None else self.seed)
        c = rng.standard_normal((self.num_topics, self.D))
        c /= np.linalg.norm(c, axis=1, keepdims=True)
        self.cs = (self.scale * c).astype(np.float32)
        if self.topics is None:
            trng = np.random.default_rng(self.seed * 7919 + self.stream)
            self.topics = trng.permutation(np.arange(self.N) % self.num_topics).astype(np.int32)
        self.key = stream_key(self.seed, self.stream)


def gen_rows_numpy(spec: RowsSpec) -> np.ndarray:
    """[N][D] float32 (or bf16 bits) rows of ``spec``."""
    i, d = np.meshgrid(np.arange(spec.N), np.arange(spec.D), indexing="ij")
    ctr = (i * spec.D + d).astype(np.uint64)
    v = element_f32(spec.cs[spec.topics][:, :], np.float32(spec.sigma), noise(spec.key, ctr))
    return v if spec.dtype == "f32" else bf16_rne(v)


def owned_mask(R: int, N: int, owned: int, seed: int) -> np.ndarray:
    """uint32 [R][ceil(N/32)]: each row owns ``owned`` blocks drawn without replacement."""
    rng = np.random.default_rng(seed)
    words = np.zeros((R, (N + 31) // 32), dtype=np.uint32)
    for r in range(R):
        j = rng.choice(N, size=owned, replace=False)
        np.bitwise_or.at(words[r], j // 32, (np.uint32(1) << (j % 32).astype(np.uint32)))
    return words


# --------------------------------------------------------------------------
# the five workloads
# --------------------------------------------------------------------------


def tiny_05b(**kw) -> CacheSpec:
    """0.5B-like: L24 H2 D64 bs16, fp32, 1 x 4096 tokens, 8 topics x2, W8 K16."""
    args = dict(name="tiny-0.5B", L=24, H=2, D=64, bs=16, dtype="f32", seq_lens=[4096],
                num_topics=8, scale=2.0, W=8, K=16, seed=1)
    args.update(kw)
    return CacheSpec(**args)


def qwen7b(**kw) -> CacheSpec:
    """7B-like: L28 H4 D128 bs128, bf16, 8 x 32768 tokens, 32 topics x1.5, W16 K32."""
    args = dict(name="7B", L=28, H=4, D=128, bs=128, dtype="bf16", seq_lens=[32768] * 8,
                num_topics=32, scale=1.5, W=16, K=32, seed=2)
    args.update(kw)
    return CacheSpec(**args)


def qwen7b_long(**kw) -> CacheSpec:
    """7B-like long context: 32 x 131072 tokens, sigma ~ U[0.5,3] per (layer, head),
    head-variance weighted, shuffled physical pages, W32 K64."""
    args = dict(name="7B-long", L=28, H=4, D=128, bs=128, dtype="bf16", seq_lens=[131072] * 32,
                num_topics=32, scale=1.5, W=32, K=64, seed=3, sigma_range=(0.5, 3.0),
                weighted=True, shuffle_pages=True)
    args.update(kw)
    return CacheSpec(**args)


def write_stress(bs: int, **kw) -> CacheSpec:
    """Prefill write path: 2^20 tokens of 7B geometry at block size ``bs``;
    topics change every 128 tokens so both block sizes hold the same Keys."""
    args = dict(name=f"write-1M-bs{bs}", L=28, H=4, D=128, bs=bs, dtype="bf16", seq_lens=[1 << 20],
                num_topics=32, scale=1.5, W=16, K=32, seed=5, span=128)
    args.update(kw)
    return CacheSpec(**args)


POOL_N, POOL_R, POOL_D, POOL_OWNED, POOL_K = 65536, 256, 128, 4096, 128


def shared_pool(N=POOL_N, R=POOL_R, D=POOL_D, owned=POOL_OWNED, K=POOL_K, seed=4):
    """Shared pool: bf16 V [N][D] (pre-pooled, noise 1/sqrt(128*28*4)),
    bf16 anchors A [R][D] (noise 1/sqrt(16*28*4)), 32 topics x1.5, and the
    ownership mask. Returns (V_spec, A_spec, mask_words, K)."""
    v = RowsSpec(N=N, D=D, num_topics=32, scale=1.5, sigma=float(np.float32(1.0 / np.sqrt(128 * 28 * 4))),
                 seed=seed, stream=2, dtype="bf16")
    a = RowsSpec(N=R, D=D, num_topics=32, scale=1.5, sigma=float(np.float32(1.0 / np.sqrt(16 * 28 * 4))),
                 seed=seed, stream=3, dtype="bf16", centroid_seed=seed)
    mask = owned_mask(R, N, owned, seed * 31 + 5)
    return v, a, mask, K


def owned_runs_mask(R: int, N: int, run: int, runs: int, seed: int) -> np.ndarray:
    """uint32 [R][ceil(N/32)]: each row owns ``runs`` whole runs of ``run``
    consecutive blocks (documents of a shared pool), drawn without replacement."""
    rng = np.random.default_rng(seed)
    n_runs = -(-N // run)
    words = np.zeros((R, (N + 31) // 32), dtype=np.uint32)
    for r in range(R):
        for d in rng.choice(n_runs, size=min(runs, n_runs), replace=False):
            j = np.arange(d * run, min(N, (d + 1) * run))
            np.bitwise_or.at(words[r], j // 32, (np.uint32(1) << (j % 32).astype(np.uint32)))
    return words


def topic_runs(N: int, num_topics: int, run: int, seed: int) -> np.ndarray:
    """int32 [N]: one random topic per run of ``run`` consecutive blocks."""
    rng = np.random.default_rng(seed)
    return np.repeat(rng.integers(0, num_topics, size=-(-N // run)), run)[:N].astype(np.int32)


HIER_POOL_DOC = 512  # blocks per document: one Grid of 8 Chunks of 64 blocks


def shared_pool_hier(N=POOL_N, R=POOL_R, D=POOL_D, docs=POOL_OWNED // HIER_POOL_DOC, K=POOL_K, seed=6):
    """Shared pool for the three-level selection: the sizes and noise of
    shared_pool, but the pool is a run of documents of HIER_POOL_DOC blocks
    whose topics change every 32 blocks, and each anchor owns ``docs`` whole
    documents (4096 blocks by default). Returns (V_spec, A_spec, mask_words, K)."""
    v = RowsSpec(N=N, D=D, num_topics=32, scale=1.5, sigma=float(np.float32(1.0 / np.sqrt(128 * 28 * 4))),
                 seed=seed, stream=2, dtype="bf16", topics=topic_runs(N, 32, 32, seed * 13 + 1))
    a = RowsSpec(N=R, D=D, num_topics=32, scale=1.5, sigma=float(np.float32(1.0 / np.sqrt(16 * 28 * 4))),
                 seed=seed, stream=3, dtype="bf16", centroid_seed=seed)
    mask = owned_runs_mask(R, N, HIER_POOL_DOC, docs, seed * 31 + 7)
    return v, a, mask, K


# --------------------------------------------------------------------------
# CUDA generator (large caches): synth/libkksynth.so
# --------------------------------------------------------------------------

_LIB = None


def _lib():
    global _LIB
    if _LIB is None:
        path = os.path.join(os.path.dirname(os.path.abspath(__file__)), "libkksynth.so")
        if not os.path.exists(path):
            raise RuntimeError(f"{path} is missing: run __graft_entry__.build() first")
        lib = ctypes.CDLL(path)
        lib.kks_gen_paged.restype = ctypes.c_int
        lib.kks_gen_paged.argtypes = [
            ctypes.c_void_p, ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_int,
            ctypes.c_longlong, ctypes.c_longlong, ctypes.c_longlong, ctypes.c_longlong,
            ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p, ctypes.c_int,
            ctypes.c_void_p, ctypes.c_void_p, ctypes.c_ulonglong, ctypes.c_void_p,
        ]
        lib.kks_gen_rows.restype = ctypes.c_int
        lib.kks_gen_rows.argtypes = [
            ctypes.c_void_p, ctypes.c_int, ctypes.c_longlong, ctypes.c_int, ctypes.c_void_p,
            ctypes.c_void_p, ctypes.c_float, ctypes.c_ulonglong, ctypes.c_void_p,
        ]
        lib.kks_fill_u32.restype = ctypes.c_int
        lib.kks_fill_u32.argtypes = [ctypes.c_void_p, ctypes.c_longlong, ctypes.c_uint, ctypes.c_void_p]
        _LIB = lib
    return _LIB


def gen_paged_cuda(spec: CacheSpec, device="cuda", storage=None):
    """Flat torch storage of the paged cache made on the GPU (same bits as
    :func:`gen_paged_numpy`). Returns the storage tensor (float32 or int16)."""
    import torch

    dt = torch.float32 if spec.dtype == "f32" else torch.int16
    n = spec.storage_elems()
    if storage is None:
        storage = torch.empty(n, dtype=dt, device=device)
    stream = torch.cuda.current_stream().cuda_stream
    lib = _lib()
    # NaN everywhere first (unused pages and the tails of partial blocks)
    if spec.dtype == "f32":
        rc = lib.kks_fill_u32(storage.data_ptr(), n, F32_NAN_BITS, stream)
    else:
        rc = lib.kks_fill_u32(storage.data_ptr(), n // 2, (BF16_NAN_BITS << 16) | BF16_NAN_BITS, stream)
        if rc == 0 and n % 2:
            storage[-1] = BF16_NAN_BITS
    if rc != 0:
        raise RuntimeError(f"kks_fill_u32 failed ({rc})")
    t = lambda a, d=torch.int32: torch.as_tensor(np.ascontiguousarray(a), dtype=d).to(device)  # noqa: E731
    pages, nv, topic, tok0 = t(spec.pages), t(spec.n_valid), t(spec.block_topic), t(spec.block_tok0, torch.int64)
    cs, sig = t(spec.cs, torch.float32), t(spec.sigma.reshape(-1), torch.float32)
    sL, sP, sH, sT = spec.strides()
    rc = lib.kks_gen_paged(
        storage.data_ptr(), 0 if spec.dtype == "f32" else 1, spec.L, spec.H, spec.D, spec.bs,
        sL, sP, sH, sT, pages.data_ptr(), nv.data_ptr(), topic.data_ptr(), tok0.data_ptr(),
        spec.total_blocks, cs.data_ptr(), sig.data_ptr(), spec.key, stream,
    )
    if rc != 0:
        raise RuntimeError(f"kks_gen_paged failed ({rc})")
    torch.cuda.current_stream().synchronize()
    return storage


def gen_rows_cuda(spec: RowsSpec, device="cuda"):
    """[N][D] rows of ``spec`` made on the GPU (float32, or int16 bf16 bits)."""
    import torch

    dt = torch.float32 if spec.dtype == "f32" else torch.int16
    out = torch.empty((spec.N, spec.D), dtype=dt, device=device)
    topic = torch.as_tensor(spec.topics, dtype=torch.int32).to(device)
    cs = torch.as_tensor(spec.cs, dtype=torch.float32).to(device)
    stream = torch.cuda.current_stream().cuda_stream
    rc = _lib().kks_gen_rows(out.data_ptr(), 0 if spec.dtype == "f32" else 1, spec.N, spec.D,
                             topic.data_ptr(), cs.data_ptr(), spec.sigma, spec.key, stream)
    if rc != 0:
        raise RuntimeError(f"kks_gen_rows failed ({rc})")
    torch.cuda.current_stream().synchronize()
    return out
