"""A CPU model of the intra kernel's data movement (csrc/gdn_prefill_tc.cu; a CTA holds 64 token
rows, 64 / C chunks, of one k-head, 256 threads): its shared-memory regions, the reach of every
M = 128 A operand (the stacked [K; Q] operand covers both tiles exactly; rows 64..127 of a W
operand read the next buffer and must stay inside the CTA's block), the tensor-memory columns
and lanes each phase uses, and which thread writes each 16-byte piece of the phase-1 q / k
tiles, the V tile, the T' / T'' tiles and, per chunk, the q / k, U image, W and P workspace
tiles: every piece exactly once and inside its buffer. The offsets and per-thread
index arithmetic are the kernel's, restated; host logic only -- the GPU parity tests check the
kernel's results against the oracle."""
import pytest

NR = 64          # token rows per CTA
THREADS = 256
NSOLVE = 128     # threads 0..127 solve; 128..255 build the V tile and copy the q / k tiles
KD = 128         # dk = dv


def kmajor_offset(r, k, K):
    return (r >> 3) * K * 16 + (k >> 3) * 128 + (r & 7) * 16 + (k & 7) * 2


def u_image_offset(r, t, C):
    return ((t >> 2) & 1) * (128 * C * 2) + kmajor_offset(r, t & ~7, C) + (t & 3) * 4


def layout(C):
    L = {}
    tile, tt = NR * KD * 2, NR * NR * 2
    L["K"], L["Q"], L["V"] = (0, tile), (tile, tile), (2 * tile, tile)
    o = 3 * tile
    for name in ("T2h", "T2l", "T1h", "T1l"):
        L[name] = (o, tt)
        o += tt
    sa = C + 4
    L["A"] = (o, NR * sa * 4); o += NR * sa * 4
    L["G"] = (o, NR * 4); o += NR * 4
    L["part"] = (o, 4 * NR * 4); o += 4 * NR * 4
    L["tok"] = (o, 3 * NR * 4); o += 3 * NR * 4   # ik, the second head's G and beta
    L["bar"] = (o, 8); o += 8
    L["tmem"] = (o, 8); o += 8
    L["t0"] = (o, 2 * (NR // C) * 4); o += 2 * (NR // C) * 4
    return L, o


def pieces_once(writes, size, what):
    """writes: byte offsets of 16-byte pieces; each in [0, size), 16-byte aligned, exactly once,
    and together covering the buffer."""
    seen = set()
    for o in writes:
        assert 0 <= o and o + 16 <= size, (what, "out of bounds", o)
        assert o % 16 == 0, (what, "misaligned", o)
        assert o not in seen, (what, "written twice", o)
        seen.add(o)
    assert len(seen) == size // 16, (what, "coverage", len(seen), size // 16)


@pytest.mark.parametrize("C", [64, 32, 16])
def test_intra_shared_memory_regions_and_operand_reach(C):
    L, total = layout(C)
    assert total <= 113 * 1024                   # two CTAs per SM
    spans = sorted(L.values())
    for (a, n), (b, _) in zip(spans, spans[1:]):
        assert a + n <= b                        # disjoint
    assert spans[-1][0] + spans[-1][1] == total
    # the stacked [K; Q] operand: rows 0..63 the k tile, 64..127 the q tile, exactly
    assert L["Q"][0] == L["K"][0] + L["K"][1] == kmajor_offset(64, 0, KD)
    assert kmajor_offset(127, KD - 1, KD) + 2 == L["K"][1] + L["Q"][1]
    # W's A operands (M = 128, K = 64): rows 64..127 read the next buffer, inside the block
    for name in ("T2h", "T2l"):
        base, size = L[name]
        last = base + kmajor_offset(127, NR - 1, NR) + 2
        assert last <= L["A"][0] and kmajor_offset(64, 0, NR) == size, name
    # exact operands: V (MN-major A, M = 128 dv, K = 64 tokens), B tiles of N = 64 rows, the
    # k tile as an MN-major B (K = 64 tokens, N = 128)
    for name, R, K in (("V", NR, KD), ("K", NR, KD), ("T1h", NR, NR), ("T1l", NR, NR)):
        base, size = L[name]
        assert kmajor_offset(R - 1, K - 1, K) + 2 == size, name
    # tensor memory (256 columns): G | QK [0, 64) (G in lanes 0..63, QK in 64..127), U^T
    # [64, 128), W [128, 256); warp w reads lanes 32 (w % 4) .. + 31
    cols = [(0, NR), (64, 64 + NR), (128, 128 + KD)]
    for (a0, a1), (b0, b1) in zip(cols, cols[1:]):
        assert a1 <= b0
    assert cols[-1][1] <= 256
    a_rows = sorted(32 * (w & 3) + l for w in range(8) if (w & 3) < 2 for l in range(32))
    p_rows = sorted(32 * (w & 3) + l - 64 for w in range(8) if (w & 3) >= 2 for l in range(32))
    for rows in (a_rows, p_rows):            # every row, in two column halves
        assert sorted(set(rows)) == list(range(NR)) and len(rows) == 2 * NR


@pytest.mark.parametrize("C", [64, 32, 16])
def test_intra_writes_cover_each_piece_once(C):
    CPC = NR // C
    L, _ = layout(C)
    # phase 1: thread (tok, which, half) writes 8 pieces of its q or k row
    q, k = [], []
    for tid in range(THREADS):
        tok, which, hf = tid & 63, (tid >> 6) & 1, tid >> 7
        for k8 in range(8):
            (k if which else q).append(kmajor_offset(tok, 64 * hf + 8 * k8, KD))
    pieces_once(q, L["Q"][1], "q tile")
    pieces_once(k, L["K"][1], "k tile")
    # V: threads NSOLVE .. 255, channel group cg, tokens 8 i + tr
    v = []
    for tid in range(NSOLVE, THREADS):
        u = tid - NSOLVE
        cg, tr = (u >> 3) & 15, u & 7
        for i in range(8):
            v.append(kmajor_offset(8 * i + tr, 8 * cg, KD))
    pieces_once(v, L["V"][1], "V tile")
    # T' / T'': solver thread tid writes row tid % 64, 8-column groups (tid // 64) + 2k of its
    # chunk's diagonal block; the rest of the tile is zeroed once per CTA when there are
    # several chunks
    diag = []
    for tid in range(NSOLVE):
        t = tid & 63
        ci = t // C
        for g in range(tid >> 6, C // 8, 2):
            diag.append(kmajor_offset(t, ci * C + 8 * g, NR))
    offdiag = [kmajor_offset(r, c, NR) for r in range(NR) for c in range(0, NR, 8)
               if r // C != c // C]
    pieces_once(diag + offdiag, L["T1h"][1], "T tile")
    assert (CPC > 1) == (len(offdiag) > 0)
    # per chunk of the CTA: U image (every warp; lane = dv row r, 32 token columns per warp),
    # W tile (warps with (w % 4) < 2; lane = token row; 64 columns per warp), P tile (the same
    # warps; row t, half of the chunk's columns)
    U = {ci: [] for ci in range(CPC)}
    W = {ci: [] for ci in range(CPC)}
    P = {ci: [] for ci in range(CPC)}
    for w in range(8):
        for lane in range(32):
            r, half = 32 * (w & 3) + lane, w >> 2
            for g in range(0, 32, 8):
                T = half * 32 + g
                ci, tu = T // C, T % C
                U[ci] += [u_image_offset(r, tu, C), u_image_offset(r, tu + 4, C)]
            if (w & 3) < 2:
                t = r
                ci, tl = t // C, t % C
                for b0 in range(0, 64, 16):
                    for e8 in (0, 8):
                        W[ci].append(kmajor_offset(tl, half * 64 + b0 + e8, KD))
            else:                              # P rows: lanes 64..127 hold QK
                t = 32 * ((w & 3) & 1) + lane
                ci, tl = t // C, t % C
                NH = C // 2
                for e8 in range(0, NH, 8):
                    P[ci].append(kmajor_offset(tl, half * NH + e8, C))
    for ci in range(CPC):
        pieces_once(U[ci], KD * C * 4, f"U image, chunk {ci}")
        pieces_once(W[ci], C * KD * 2, f"W tile, chunk {ci}")
        pieces_once(P[ci], C * C * 2, f"P tile, chunk {ci}")
    # q / k tiles -> workspace: threads NSOLVE .. 255 after the V tile, each chunk's contiguous
    # slice
    nthr = THREADS - NSOLVE
    for ci in range(CPC):
        slice_pieces = C * KD * 2 // 16
        got = [16 * i for u in range(nthr) for i in range(u, slice_pieces, nthr)]
        pieces_once(got, C * KD * 2, f"q / k workspace tile, chunk {ci}")
        assert (ci + 1) * C * KD * 2 <= L["K"][1]


def test_pass_state_handoff_layout():
    """The state pass hands a (sequence, value head)'s fp32 state to the next piece through a 64 KB
    block: compute thread (row r = 32 (w % 4) + lane, half = w // 4) stores and loads float4 piece j
    (dk columns 4 (16 half + j) .. + 3) at float offset ((16 half + j) * 128 + r) * 4. Every element
    once, inside the block, at the same place for the store and the load; and at each step j a
    warp's 32 rows cover 512 contiguous bytes."""
    seen = {}
    for w in range(8):
        half = w >> 2
        steps = {}
        for lane in range(32):
            r = 32 * (w & 3) + lane
            for j in range(16):
                off = ((half * 16 + j) * 128 + r) * 4
                assert 0 <= off and off + 4 <= 128 * 128
                for e in range(4):
                    elem = (r, 4 * (half * 16 + j) + e)
                    assert off + e not in seen, "two elements at one place"
                    seen[off + e] = elem
                steps.setdefault(j, []).append(off * 4)
        for j, byte_offs in steps.items():
            byte_offs.sort()
            assert byte_offs[-1] - byte_offs[0] == 31 * 16       # 32 rows, 16 bytes each, contiguous
            assert all(b - a == 16 for a, b in zip(byte_offs, byte_offs[1:]))
    assert len(seen) == 128 * 128
    assert sorted(seen.values()) == [(r, c) for r in range(128) for c in range(128)]
