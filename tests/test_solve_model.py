"""A CPU model of the intra kernel's triangular solve (csrc/gdn_prefill_tc.cu; a CTA holds 64
token rows, 64 / C chunks, solved by 128 threads): the same per-thread index arithmetic over the
fp32 A / T rows of stride C + 4 (four padding floats per row), every shared-memory access checked
for bounds, 16-byte alignment of the vector accesses and reads of initialised data only, with the
kernel's barriers at the same points (each phase reads everything first, then writes, as the
barrier between them allows). The solve is a blocked recursive inverse: 8 x 8 diagonal blocks by
forward substitution, then blocks of 16, 32 and 64 rows (as far as the chunk goes) from two
halves, T21 = -T22 (A21 T11). The result T must equal (I + A)^-1 per chunk; a planted index
mistake fails. The model is host logic only; the GPU parity tests check the kernel itself against
the oracle."""
import numpy as np
import pytest

NROW = 64        # token rows per intra CTA
NSOLVE = 128     # solver threads (warps 0-3)


def merge_threads(b):
    """(active threads, rows per thread) of the merge that builds blocks of 2b rows."""
    rb = 2 if b == 32 else 1
    return (NROW // (2 * b)) * b * b // (4 * rb), rb


def run_model(C, seed=0, mutant=None):
    SA = C + 4
    sA = np.full(NROW * SA, np.nan, dtype=np.float64)   # NaN = never written

    def rd(i):
        assert 0 <= i < NROW * SA, ("read oob", i)
        v = sA[i]
        assert not np.isnan(v), ("read unwritten", i)
        return v

    def wr(i, v):
        assert 0 <= i < NROW * SA, ("write oob", i)
        sA[i] = v

    def rd4(i):
        assert i % 4 == 0, ("float4 misaligned", i)
        return np.array([rd(i + k) for k in range(4)])

    def wr4(i, v):
        assert i % 4 == 0, ("float4 misaligned", i)
        for k in range(4):
            wr(i + k, v[k])

    rng = np.random.default_rng(seed)
    CPC = NROW // C
    A = np.zeros((CPC, C, C))
    for ci in range(CPC):
        A[ci] = np.tril(rng.standard_normal((C, C)) * 0.3, -1)
    # A/P phase: thread (row t, half) writes its C / 2 columns as float4 (row-contiguous)
    NH = C // 2
    for t in range(NROW):
        ci, tl = divmod(t, C)
        for half in range(2):
            for k in range(NH // 4):
                j0 = half * NH + 4 * k
                wr4(t * SA + j0, A[ci][tl][j0:j0 + 4])
        wr4(t * SA + C, [0.5] * 4)   # padding (scale, beta, iq, ik), not read by the solve

    # level 0: 8 x 8 diagonal blocks, thread = (block, column c): threads 0..63
    writes = []
    for tid in range(NSOLVE):
        if tid >= 64:
            continue
        R0 = 8 * (tid >> 3)
        c = tid & 7
        o = R0 % C
        x = [0.0] * 8
        for r in range(8):
            a = np.concatenate([rd4((R0 + r) * SA + o), rd4((R0 + r) * SA + o + 4)])
            s0 = s1 = 0.0
            for l in range(0, r, 2):
                s0 += a[l] * x[l]
                if l + 1 < r:
                    s1 += a[l + 1] * x[l + 1]
            x[r] = 0.0 if r < c else (1.0 if r == c else -(s0 + s1))
        for r in range(8):
            writes.append(((R0 + r) * SA + o + c, x[r]))
    for i, v in writes:                        # after the barrier: in place
        wr(i, v)

    # merges: blocks of 2b rows from two b-row halves
    b = 8
    while 2 * b <= C:
        nt, rb = merge_threads(b)
        per_merge = b * b // (4 * rb)
        cols = b // 4
        # X = A21 T11 (T11 is lower triangular: column block j0 needs l >= j0)
        res = []
        for tid in range(nt):
            m, idx = divmod(tid, per_merge)
            R0 = 2 * b * m
            o = R0 % C
            j0 = 4 * (idx % cols)
            i0 = rb * (idx // cols)
            if mutant == "X from l = 0 of the next half":
                j0_l = j0 + 4 if j0 + 4 < b else j0
            else:
                j0_l = j0
            acc = np.zeros((rb, 4))
            for l in range(j0_l, b, 4):
                av = [rd4((R0 + b + i0 + i) * SA + o + l) for i in range(rb)]
                tv = [rd4((R0 + l + kk) * SA + o + j0) for kk in range(4)]
                for i in range(rb):
                    for kk in range(4):
                        acc[i] += av[i][kk] * tv[kk]
            res.append((R0, o, i0, j0, acc))
        for R0, o, i0, j0, acc in res:         # after the barrier: X over A21
            for i in range(rb):
                wr4((R0 + b + i0 + i) * SA + o + j0, acc[i])
        # T21 = -(T22 X) (T22 is lower triangular: rows i0 .. i0 + rb - 1 need l < i0 + rb)
        res = []
        for tid in range(nt):
            m, idx = divmod(tid, per_merge)
            R0 = 2 * b * m
            o = R0 % C
            j0 = 4 * (idx % cols)
            i0 = rb * (idx // cols)
            acc = np.zeros((rb, 4))
            for l in range(0, i0 + rb, 4):
                av = [rd4((R0 + b + i0 + i) * SA + o + b + l) for i in range(rb)]
                xv = [rd4((R0 + b + l + kk) * SA + o + j0) for kk in range(4)]
                for i in range(rb):
                    for kk in range(4):
                        acc[i] += av[i][kk] * xv[kk]
            res.append((R0, o, i0, j0, -acc))
        for R0, o, i0, j0, acc in res:         # after the barrier: T21 over X
            for i in range(rb):
                wr4((R0 + b + i0 + i) * SA + o + j0, acc[i])
        b *= 2

    # the T' / T'' step reads rows: T[t][8g .. 8g+7], thread t % 64, groups (t >> 6) + 2k
    for tid in range(NSOLVE):
        t = tid & 63
        for g in range(tid >> 6, C // 8, 2):
            rd4(t * SA + 8 * g)
            rd4(t * SA + 8 * g + 4)
    ok = True
    for ci in range(CPC):
        T = np.zeros((C, C))
        for r in range(C):
            for g in range(C // 8):
                T[r, 8 * g:8 * g + 8] = np.concatenate(
                    [rd4((ci * C + r) * SA + 8 * g), rd4((ci * C + r) * SA + 8 * g + 4)])
        ref = np.linalg.inv(np.eye(C) + A[ci])
        ok &= np.abs(T - ref).max() / np.abs(ref).max() < 1e-12
    return ok


@pytest.mark.parametrize("C", [64, 32, 16])
def test_solve_model_inverse_and_accesses(C):
    assert run_model(C, seed=C)


def test_solve_model_threads_fit():
    for b in (8, 16, 32):
        nt, rb = merge_threads(b)
        assert nt <= NSOLVE and nt % 32 == 0
        assert nt * 4 * rb == (NROW // (2 * b)) * b * b   # every output exactly once


def test_solve_model_catches_a_planted_mistake():
    """Skipping the first column block of T11 in X = A21 T11 gives a wrong T."""
    assert not run_model(64, seed=1, mutant="X from l = 0 of the next half")
