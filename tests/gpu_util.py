"""Helpers for the GPU parity tests: put seeded storage on the device, run the
C ABI, read C back (with canary guard bands around it), and compare with the
oracle under the acceptance rules."""

from __future__ import annotations

import numpy as np

import datagen
import dense_gemm_06_gb300 as lg
import oracle
from acceptance import assert_accepted

CANARY = {"f32": np.array([0x7FC0BEEF], np.uint32).view(np.float32)[0],
          "f16": np.uint16(0x7E5A), "bf16": np.uint16(0x7FDA)}
GUARD = 64  # elements before and after C


def torch_mod():
    import torch
    return torch


def to_device(storage: np.ndarray):
    torch = torch_mod()
    if storage.dtype == np.uint16:
        return torch.from_numpy(storage.view(np.int16).copy()).cuda()
    return torch.from_numpy(storage.copy()).cuda()


def decode(raw: np.ndarray, t: str) -> np.ndarray:
    if t == "f32":
        return raw.view(np.float32).astype(np.float64)
    if t == "f16":
        return raw.view(np.float16).astype(np.float64)
    return (raw.view(np.uint16).astype(np.uint32) << np.uint32(16)).view(np.float32).astype(np.float64)


class CBuffer:
    """C storage on the device with guard bands and canary-filled padding."""

    def __init__(self, M, N, c_major, ldc, ot):
        self.M, self.N, self.c_major, self.ldc, self.ot = M, N, c_major, ldc, ot
        inner, outer = (N, M) if c_major == lg.GEMM_MAJOR_MN else (M, N)
        self.inner, self.outer = inner, outer
        self.span = 0 if inner == 0 or outer == 0 else (outer - 1) * ldc + inner
        np_t = np.float32 if ot == "f32" else np.uint16
        host = np.empty(self.span + 2 * GUARD, dtype=np_t)
        host[:] = CANARY[ot]
        self.host_init = host
        self.dev = to_device(host)
        self.esize = 4 if ot == "f32" else 2

    def ptr(self) -> int:
        return int(self.dev.data_ptr()) + GUARD * self.esize

    def fill(self, logical_storage: np.ndarray):
        """Write a logical (M x N) matrix of C's storage type into the body
        (padding and guard bands keep their canaries); returns the storage
        array of the body as the C ABI addresses it."""
        torch = torch_mod()
        host = self.host_init.copy()
        body = host[GUARD:GUARD + self.span]
        L = logical_storage if self.c_major == lg.GEMM_MAJOR_MN else logical_storage.T
        for r in range(self.outer):
            body[r * self.ldc:r * self.ldc + self.inner] = L[r]
        self.host_init = host  # canaries of padding/guards unchanged
        src = host.view(np.int16) if host.dtype == np.uint16 else host
        self.dev.copy_(torch.from_numpy(src.copy()).to(self.dev.device))
        return body.copy()

    def read(self) -> np.ndarray:
        """Logical C (M x N, float64); asserts guard bands and padding intact."""
        raw = self.dev.cpu().numpy()
        raw = raw.view(np.float32) if self.ot == "f32" else raw.view(np.uint16)
        init = self.host_init
        assert np.array_equal(raw[:GUARD].view(np.uint8), init[:GUARD].view(np.uint8)), \
            "C guard band before the matrix was overwritten"
        assert np.array_equal(raw[GUARD + self.span:].view(np.uint8),
                              init[GUARD + self.span:].view(np.uint8)), \
            "C guard band after the matrix was overwritten"
        body = raw[GUARD:GUARD + self.span]
        if self.span == 0:
            return np.zeros((self.M, self.N))
        full = np.empty(self.outer * self.ldc, dtype=body.dtype)
        full[:self.span] = body
        full[self.span:] = init[0]
        grid = full.reshape(self.outer, self.ldc)
        if self.ldc > self.inner:
            pad = grid[:, self.inner:]
            assert np.array_equal(pad.view(np.uint8),
                                  np.full_like(pad, init[0]).view(np.uint8)), \
                "padding between rows of C was overwritten"
        vals = decode(np.ascontiguousarray(grid[:, :self.inner]), self.ot)
        return vals if self.c_major == lg.GEMM_MAJOR_MN else vals.T.copy()


def make_operands(M, N, K, dtype, a_major, b_major, dist, seed, lda_pad=0, ldb_pad=0,
                  lo=-5, hi=5):
    it = lg.IN_TYPE[dtype]
    lda = (K if a_major == 0 else M) + lda_pad
    ldb = (K if b_major == 0 else N) + ldb_pad
    A = datagen.operand(M, K, major=a_major, ld=lda, dtype=it, dist=dist, seed=seed,
                        stream=0, lo=lo, hi=hi)
    B = datagen.operand(N, K, major=b_major, ld=ldb, dtype=it, dist=dist, seed=seed,
                        stream=1, lo=lo, hi=hi)
    return A, lda, B, ldb


def run_device_gemm(M, N, K, dtype, A, lda, a_major, B, ldb, b_major, c_major=1, ldc_pad=0,
                    cta_group=0, dA=None, dB=None, tc_store=0, multicast=0, scheduler=0,
                    tile_n=0, split=0):
    """Runs gemm() through the C ABI; returns the logical C (float64)."""
    torch = torch_mod()
    ot = lg.OUT_TYPE[dtype]
    ldc = (N if c_major == lg.GEMM_MAJOR_MN else M) + ldc_pad
    if dA is None:
        dA = to_device(A) if A.size else None
    if dB is None:
        dB = to_device(B) if B.size else None
    cbuf = CBuffer(M, N, c_major, ldc, ot)
    old = lg.gemm_get_option(lg.GEMM_OPT_TC_CTA_GROUP)
    old_store = lg.gemm_get_option(lg.GEMM_OPT_TC_STORE)
    old_mc = lg.gemm_get_option(lg.GEMM_OPT_TC_MULTICAST)
    old_sched = lg.gemm_get_option(lg.GEMM_OPT_TC_SCHEDULER)
    old_tile = lg.gemm_get_option(lg.GEMM_OPT_TC_TILE_N)
    old_split = lg.gemm_get_option(lg.GEMM_OPT_TC_SPLIT_TAIL)
    lg.check(lg.gemm_set_option(lg.GEMM_OPT_TC_TILE_N, tile_n), "set_option")
    lg.check(lg.gemm_set_option(lg.GEMM_OPT_TC_SPLIT_TAIL, split), "set_option")
    lg.check(lg.gemm_set_option(lg.GEMM_OPT_TC_CTA_GROUP, cta_group), "set_option")
    lg.check(lg.gemm_set_option(lg.GEMM_OPT_TC_STORE, tc_store), "set_option")
    lg.check(lg.gemm_set_option(lg.GEMM_OPT_TC_MULTICAST, multicast), "set_option")
    lg.check(lg.gemm_set_option(lg.GEMM_OPT_TC_SCHEDULER, scheduler), "set_option")
    try:
        rc = lg.gemm(M, N, K, dA if dA is not None else 0, lda, a_major,
                     dB if dB is not None else 0, ldb, b_major, cbuf.ptr(), ldc, c_major, dtype)
        lg.check(rc, "gemm")
        lg.check(lg.gemm_check_device_error(), "device error word")
        torch.cuda.synchronize()
    finally:
        lg.gemm_set_option(lg.GEMM_OPT_TC_CTA_GROUP, old)
        lg.gemm_set_option(lg.GEMM_OPT_TC_STORE, old_store)
        lg.gemm_set_option(lg.GEMM_OPT_TC_MULTICAST, old_mc)
        lg.gemm_set_option(lg.GEMM_OPT_TC_SCHEDULER, old_sched)
        lg.gemm_set_option(lg.GEMM_OPT_TC_TILE_N, old_tile)
        lg.gemm_set_option(lg.GEMM_OPT_TC_SPLIT_TAIL, old_split)
    return cbuf.read()


def check_full(C, M, N, K, dtype, A, lda, a_major, B, ldb, b_major, exact, what):
    it, ot = lg.IN_TYPE[dtype], lg.OUT_TYPE[dtype]
    C_ref, S = oracle.gemm_ref(M, N, K, A, lda, a_major, it, B, ldb, b_major, it)
    return assert_accepted(C, C_ref, S, ot, exact=exact, what=what)


def check_sampled(C, M, N, K, dtype, A, lda, a_major, B, ldb, b_major, exact, what, seed,
                  count=256):
    """256 seeded rows (all columns) and 256 seeded columns (all rows), plus
    the first and last row/column."""
    it, ot = lg.IN_TYPE[dtype], lg.OUT_TYPE[dtype]
    rows = datagen.sample_indices(M, count, seed=seed + 1, stream=101)
    cols = datagen.sample_indices(N, count, seed=seed + 1, stream=102)
    Cr, Sr = oracle.gemm_ref(M, N, K, A, lda, a_major, it, B, ldb, b_major, it, rows=rows)
    w1 = assert_accepted(C[rows, :], Cr, Sr, ot, exact=exact, what=what + " (sampled rows)")
    Cc, Sc = oracle.gemm_ref(M, N, K, A, lda, a_major, it, B, ldb, b_major, it, cols=cols)
    w2 = assert_accepted(C[:, cols], Cc, Sc, ot, exact=exact, what=what + " (sampled cols)")
    return max(w1, w2)
