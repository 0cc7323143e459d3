"""Shared helpers of the GPU parity tests: device copies of synthetic caches,
the tolerances of the method's acceptance bar, and the top-K set criterion."""
from __future__ import annotations

import numpy as np
import torch

import synth

# Acceptance bar: pooled vectors and anchors agree with the oracle within
# 1e-5 of the vector's largest magnitude (normwise, since an element-wise
# relative bound is ill-posed near zero); scores within 1e-5 relative (with a
# floor of 1e-3 on the magnitude); top-K sets agree except for swaps between
# candidates whose oracle scores are within 1e-6 of each other.
VEC_RTOL = 1e-5
SCORE_RTOL = 1e-5
TIE_EPS = 1e-6


def assert_vec_close(gpu, ref, what=""):
    gpu = np.asarray(gpu, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    assert gpu.shape == ref.shape, (gpu.shape, ref.shape)
    scale = np.max(np.abs(ref), axis=-1, keepdims=True)
    err = np.max(np.abs(gpu - ref), axis=-1, keepdims=True)
    bad = err > VEC_RTOL * scale + (scale == 0) * 0.0
    if np.any(bad):
        i = np.argwhere(bad)[0]
        raise AssertionError(f"{what}: vector {tuple(i)} err {err[tuple(i)]} > {VEC_RTOL} * {scale[tuple(i)]}")


def assert_scores_close(gpu, ref, what=""):
    gpu = np.asarray(gpu, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    tol = SCORE_RTOL * np.maximum(np.abs(ref), 1e-3)
    bad = np.abs(gpu - ref) > tol
    if np.any(bad):
        i = np.flatnonzero(bad.reshape(-1))[0]
        raise AssertionError(f"{what}: score {i}: gpu {gpu.reshape(-1)[i]} oracle {ref.reshape(-1)[i]}")


def assert_topk_valid(gpu_idx, gpu_top, oracle_scores, K, what=""):
    """GPU top-K of one request against the oracle's scores of every candidate.

    The GPU set must hold every candidate whose oracle score beats the oracle's
    K-th score by more than TIE_EPS, and only candidates within TIE_EPS of it
    or above; the listed scores must be non-increasing and match the oracle's;
    missing slots are -1 / -inf.
    """
    s = np.asarray(oracle_scores, dtype=np.float64)
    gpu_idx = np.asarray(gpu_idx).astype(np.int64)
    n = len(s)
    k = min(K, n)
    assert np.all(gpu_idx[k:] == -1), f"{what}: slots past {k} not empty"
    if gpu_top is not None:
        assert np.all(np.isneginf(np.asarray(gpu_top)[k:])), f"{what}: scores past {k} not -inf"
    if k == 0:
        return
    sel = gpu_idx[:k]
    assert np.all((sel >= 0) & (sel < n)), f"{what}: index out of range {sel}"
    assert len(set(sel.tolist())) == k, f"{what}: duplicate indices"
    sK = np.sort(s)[::-1][k - 1]
    must = set(np.flatnonzero(s > sK + TIE_EPS).tolist())
    missing = must - set(sel.tolist())
    assert not missing, f"{what}: missing {sorted(missing)[:5]} (K-th score {sK})"
    assert np.all(s[sel] >= sK - TIE_EPS), f"{what}: selected below the K-th score"
    if gpu_top is not None:
        top = np.asarray(gpu_top, dtype=np.float64)[:k]
        assert np.all(np.diff(top) <= 0), f"{what}: scores not descending"
        assert_scores_close(top, s[sel], what + " top scores")


class DeviceCache:
    """A synthetic paged cache on the GPU with its block table and descriptor."""

    def __init__(self, spec: synth.CacheSpec, device="cuda"):
        from kv_cache_block_gb300 import kk

        self.spec = spec
        self.storage = synth.gen_paged_cuda(spec, device=device)
        self.desc = kk.kcache_desc(self.storage, kk.KK_F32 if spec.dtype == "f32" else kk.KK_BF16,
                                   spec.L, spec.H, spec.D, spec.bs, spec.num_pages, spec.strides())
        t = lambda a: torch.as_tensor(np.ascontiguousarray(a), dtype=torch.int32).to(device)  # noqa: E731
        self.pages = t(spec.pages)
        self.offsets = t(spec.offsets)
        self.seq_lens = t(spec.seq_lens)
        self.n_valid = t(spec.n_valid)
        self.bt = kk.BlockTable(self.pages, self.offsets, self.seq_lens, max(spec.nb) if spec.nb else 0)

    def host_view(self):
        """numpy [L][P][H][bs][D] view of the whole cache (small caches only)."""
        arr = self.storage.cpu().numpy()
        if self.spec.dtype == "bf16":
            arr = arr.view(np.uint16)
        return synth.view_paged(arr, self.spec)

    def host_pages(self, pages):
        """numpy [L][len(pages)][H][bs][D] copy of a few physical pages."""
        sp = self.spec
        L, P, H, bs, D = sp.shape
        idx = torch.as_tensor(np.asarray(pages, dtype=np.int64), device=self.storage.device)
        if sp.layout == "LPHTD":
            t = self.storage.view(L, P, H, bs, D).index_select(1, idx)
        elif sp.layout == "PLHTD":
            t = self.storage.view(P, L, H, bs, D).index_select(0, idx).transpose(0, 1)
        else:
            t = self.storage.view(L, P, bs, H, D).index_select(1, idx).transpose(2, 3)
        arr = t.contiguous().cpu().numpy()
        return arr.view(np.uint16) if sp.dtype == "bf16" else arr

    def host_request(self, r):
        """(numpy cache view holding only request r's pages, remapped page list)."""
        pr = self.spec.pages_of(r)
        return self.host_pages(pr), np.arange(len(pr))
