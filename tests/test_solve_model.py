"""A CPU model of the intra kernel's triangular solve (csrc/gdn_prefill_tc.cu; a CTA holds 64
token rows, 64 / C chunks, solved by 64 threads): the same per-thread index arithmetic over the
fp32 A / T rows of stride C + 4 (four padding floats per row), every shared-memory access checked for bounds, 16-byte alignment of the vector accesses
and reads of initialised data only, with the kernel's barriers at the same points. The result
T must equal (I + A)^-1 per chunk. The model is host logic only; the GPU parity tests check the
kernel itself against the oracle."""
import numpy as np
import pytest

NROW = 64        # token rows per intra CTA
NSOLVE = 64      # solver threads (warps 0-1)


def run_model(C, seed=0):
    SA = C + 4
    sA = np.full(NROW * SA, np.nan, dtype=np.float64)   # NaN = never written
    def rd(i):
        assert 0 <= i < NROW * SA, ("read oob", i); v = sA[i]; assert not np.isnan(v), ("read unwritten", i); return v
    def wr(i, v):
        assert 0 <= i < NROW * SA, ("write oob", i); sA[i] = v
    def rd4(i):
        assert i % 4 == 0, ("float4 misaligned", i); return [rd(i + k) for k in range(4)]
    rng = np.random.default_rng(seed)
    CPC = NROW // C
    A = np.zeros((CPC, C, C))
    for ci in range(CPC):
        M = rng.standard_normal((C, C)) * 0.3
        A[ci] = np.tril(M, -1)
    # A/P phase: thread (row t, half) writes its NH columns as float4 (row-contiguous)
    NH = C // 2
    for t in range(NROW):
        ci, tl = divmod(t, C)
        for half in range(2):
            for k in range(NH // 4):
                j0 = half * NH + 4 * k
                for e in range(4):
                    wr(t * SA + j0 + e, A[ci][tl][j0 + e])
        for k in range(4):
            wr(t * SA + C + k, 0.5)   # padding (scale, beta, iq, ik), not read by the solve
    # step 1: diagonal blocks of B1 rows, thread = (block, column c)
    B1 = min(C, 32)
    X1 = {}
    for tid in range(NSOLVE):
        row0 = (tid // B1) * B1; c = tid % B1; o = row0 % C
        base = row0 * SA + o
        x = [0.0] * B1
        for r in range(B1):
            s0 = s1 = 0.0
            for l4 in range(0, r, 4):
                a4 = rd4(base + r * SA + l4)
                s0 += a4[0] * x[l4]
                if l4 + 1 < r: s1 += a4[1] * x[l4 + 1]
                if l4 + 2 < r: s0 += a4[2] * x[l4 + 2]
                if l4 + 3 < r: s1 += a4[3] * x[l4 + 3]
            x[r] = 0.0 if r < c else (1.0 if r == c else -(s0 + s1))
        X1[tid] = (base, c, x)
    for tid, (base, c, x) in X1.items():      # after the barrier: in place
        for r in range(B1):
            wr(base + r * SA + c, x[r])
    if C == 64:
        # step 2a: X = A21 T11, 64 threads, 4x4 outputs per thread
        res = {}
        for tid in range(NSOLVE):
            k = tid
            r0 = 4 * (k >> 3); c0 = 4 * (k & 7)
            cb = 0
            acc = np.zeros((4, 4))
            for l in range(0, 32, 4):
                a = [rd4(cb + (32 + r0 + i) * SA + l) for i in range(4)]
                tt = [rd4(cb + (l + kk) * SA + c0) for kk in range(4)]
                for i in range(4):
                    for kk in range(4):
                        for jj in range(4):
                            acc[i][jj] += a[i][kk] * tt[kk][jj]
            res[tid] = (cb, r0, c0, acc)
        for tid, (cb, r0, c0, acc) in res.items():   # after the barrier: X over A21
            for i in range(4):
                for jj in range(4):
                    wr(cb + (32 + r0 + i) * SA + c0 + jj, acc[i][jj])
        # step 2b: T21 = -(T22 X), l < r0 + 4 (T22 rows r0..r0+3 are zero beyond)
        res = {}
        for tid in range(NSOLVE):
            k = tid
            r0 = 4 * (k >> 3); c0 = 4 * (k & 7)
            cb = 0
            acc = np.zeros((4, 4))
            for l in range(0, r0 + 4, 4):
                a = [rd4(cb + (32 + r0 + i) * SA + 32 + l) for i in range(4)]
                xx = [rd4(cb + (32 + l + kk) * SA + c0) for kk in range(4)]
                for i in range(4):
                    for kk in range(4):
                        for jj in range(4):
                            acc[i][jj] += a[i][kk] * xx[kk][jj]
            res[tid] = (cb, r0, c0, -acc)
        for tid, (cb, r0, c0, acc) in res.items():
            for i in range(4):
                for jj in range(4):
                    wr(cb + (32 + r0 + i) * SA + c0 + jj, acc[i][jj])
    # step 3 reads rows: T[t][8g .. 8g+7]
    ok = True
    for ci in range(CPC):
        T = np.zeros((C, C))
        for r in range(C):
            for g in range(C // 8):
                v = rd4(ci * C * SA + r * SA + 8 * g) + rd4(ci * C * SA + r * SA + 8 * g + 4)
                T[r, 8 * g:8 * g + 8] = v
        ref = np.linalg.inv(np.eye(C) + A[ci])
        err = np.abs(T - ref).max() / np.abs(ref).max()
        ok &= err < 1e-12
    return ok


@pytest.mark.parametrize("C", [64, 32, 16])
def test_solve_model_inverse_and_accesses(C):
    assert run_model(C, seed=C)
