"""Pins of the fp64 CPU oracle against what the pages and the mathematics fix.

None of these checks retypes the oracle's formulas: each compares it with a
worked value from the bf16 format, a library routine (torch's fp32 -> bf16
cast, complex exponentials, numpy matmul), an exact rational computation, a
closed form or invariant stated on the pages, or a brute-force restatement
written differently (tests/_indep.py).

Page citations (gist.science summaries):
  Leyline §2.1 (directive), §2.2 (Δ = |R|-|S|, K_pe_new = R(Δ)K_pe,
  R(a)R(b) = R(a+b), unitary rotation), §2.3 (downstream re-indexing),
  §4.3 (drift ≈ 4.7e-3 relative L2 in bf16);
  Irminsul §2.1 (cKV 512 verbatim = 89% of the row, k_r 64 = 11%), §2.2
  (δ = p_target - p_source), §3 (4.7e-3 relative L2);
  Kamera §2 (R(δ)KV(B|∅) + U_m V_mᵀ; byte-for-byte c_KV reuse).
"""
import math
import os

import numpy as np
import pytest
import torch

import _indep as ind
import oracle as O
import synth

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")
BASES = (10000.0, 500000.0)


# ---------------------------------------------------------------------------
# bf16 rounding
# ---------------------------------------------------------------------------

def _golden_rne():
    rows = []
    with open(os.path.join(GOLDEN, "bf16_rne.txt")) as f:
        for line in f:
            if line.startswith("#") or not line.strip():
                continue
            a, b = line.split()[:2]
            rows.append((float.fromhex(a), int(b, 16)))
    return rows


@pytest.mark.parametrize("v,want", _golden_rne())
def test_round_bf16_worked_values(oracle, v, want):
    assert oracle.round_bf16(v) == want
    assert ind.round_bf16(v) == want


def test_round_bf16_matches_torch_on_fp32_inputs(oracle):
    # torch's fp32 -> bf16 cast rounds to nearest even; on inputs that are
    # already fp32 a direct fp64 -> bf16 rounding must agree with it.
    rng = np.random.default_rng(7)
    f = rng.standard_normal(20000).astype(np.float32) * np.float32(10.0) ** rng.integers(
        -30, 30, 20000).astype(np.float32)
    # plus exact ties: a bf16 value plus half its ulp
    b = (rng.integers(0, 0x7F00, 4000).astype(np.uint32) << 16)
    ties = (b | 0x8000).view(np.float32)
    f = np.concatenate([f, ties, -ties]).astype(np.float32)
    f = f[np.isfinite(f)]
    want = torch.from_numpy(f).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    got = oracle.round_bf16_array(f.astype(np.float64))
    assert np.array_equal(got, want)


def test_round_bf16_matches_exact_rationals(oracle):
    rng = np.random.default_rng(11)
    v = rng.standard_normal(3000) * np.exp2(rng.integers(-140, 130, 3000).astype(np.float64))
    got = oracle.round_bf16_array(v)
    want = np.array([ind.round_bf16(float(x)) for x in v], dtype=np.uint16)
    assert np.array_equal(got, want)


def test_round_bf16_is_not_double_rounding(oracle):
    # 1 + 2^-8 + 2^-40 lies just above a bf16 tie; rounding it to fp32 first
    # lands exactly on the tie and would then round down.
    v = 1.0 + 2.0 ** -8 + 2.0 ** -40
    via_f32 = torch.tensor([v], dtype=torch.float32).to(torch.bfloat16).view(torch.int16).item()
    assert via_f32 & 0xFFFF == 0x3F80
    assert oracle.round_bf16(v) == 0x3F81


def test_bf16_widening_is_exact(oracle):
    b = np.arange(0, 65536, dtype=np.uint32).astype(np.uint16)
    want = torch.from_numpy(b.view(np.int16)).view(torch.bfloat16).to(torch.float64).numpy()
    got = oracle.bf16_to_f64(b)
    fin = np.isfinite(want)
    assert np.array_equal(got[fin], want[fin])
    assert np.array_equal(np.isnan(got), np.isnan(want))


# ---------------------------------------------------------------------------
# The rotation R(δ)
# ---------------------------------------------------------------------------

@pytest.mark.parametrize("base,d", [(10000.0, 64), (500000.0, 128), (10000.0, 8)])
def test_rotation_is_complex_multiplication(oracle, base, d):
    # rotate-half pairing: z_j = x[j] + i x[j+d/2] turned by exp(i δ θ_j)
    rng = np.random.default_rng(3)
    h = d // 2
    th = base ** (-2.0 * np.arange(h) / d)
    for delta in (1, -1, 7, -1008, 32768, -32768, 100000, -100000, 65536):
        x = rng.standard_normal(d)
        y = oracle.rotate_f64(x, delta, base)
        z = (x[:h] + 1j * x[h:]) * np.exp(1j * (delta * th))
        # numpy's vectorised pow may differ from libm's by an ulp in θ_j,
        # which moves the angle δθ_j by up to ~|δ|·2^-52
        tol = 1e-14 + 8 * 2.0 ** -52 * abs(delta) * np.max(np.abs(x))
        assert np.allclose(y[:h], z.real, rtol=0, atol=tol)
        assert np.allclose(y[h:], z.imag, rtol=0, atol=tol)


def test_pair_zero_is_a_plain_2d_rotation(oracle):
    # θ_0 = 1, so pair 0 turns by δ radians, counter-clockwise for δ > 0
    for delta in (1, 2, -3, 1000):
        x = np.zeros(64)
        x[0] = 1.0
        y = oracle.rotate_f64(x, delta, 10000.0)
        assert y[0] == pytest.approx(math.cos(delta), abs=1e-15)
        assert y[32] == pytest.approx(math.sin(delta), abs=1e-15)


@pytest.mark.parametrize("base,d", [(10000.0, 64), (500000.0, 128)])
def test_frequencies_are_geometric(oracle, base, d):
    # angle turned by pair j under R(1), read back with atan2: θ_j = base^(-2j/d)
    h = d // 2
    ang = []
    for j in range(h):
        x = np.zeros(d)
        x[j] = 1.0
        y = oracle.rotate_f64(x, 1, base)
        ang.append(math.atan2(y[j + h], y[j]))
    ang = np.array(ang)
    assert ang[0] == pytest.approx(1.0, abs=1e-15)
    ratio = ang[1:] / ang[:-1]
    assert np.allclose(ratio, base ** (-2.0 / d), rtol=1e-12)
    assert oracle.theta(base, 0, d) == 1.0


def test_one_hot_pairing(oracle):
    # a single nonzero input element only ever reaches itself and its partner j ± d/2
    d, h = 64, 32
    for j0 in (0, 5, 31, 32, 40, 63):
        x = np.zeros(d)
        x[j0] = 1.0
        y = oracle.rotate_f64(x, 12345, 10000.0)
        nz = set(np.nonzero(np.abs(y) > 0)[0].tolist())
        assert nz <= {j0, (j0 + h) % d}


@pytest.mark.parametrize("base,d", [(10000.0, 64), (500000.0, 128)])
def test_closure(oracle, base, d):
    # R(a)R(b) = R(a+b) and R(δ)R(-δ) = I (Leyline §2.2).  The fp64 angle δθ
    # carries a relative error of ~1e-16, i.e. up to ~3e-11 rad at |δ| ~ 1e5.
    rng = np.random.default_rng(5)
    shifts = [1, -1, 1000, -1000, 32768, -32768, 100000, -100000] + list(
        rng.integers(-100000, 100001, 8))
    for a in shifts:
        for b in shifts[::3]:
            x = rng.standard_normal(d)
            ab = oracle.rotate_f64(oracle.rotate_f64(x, a, base), b, base)
            direct = oracle.rotate_f64(x, int(a) + int(b), base)
            assert np.max(np.abs(ab - direct)) <= 1e-9 * np.linalg.norm(x)
        x = rng.standard_normal(d)
        back = oracle.rotate_f64(oracle.rotate_f64(x, a, base), -int(a), base)
        assert np.max(np.abs(back - x)) <= 1e-9 * np.linalg.norm(x)


def test_attention_scores_depend_on_relative_position(oracle):
    # ⟨R(a)q, R(b)k⟩ = ⟨R(a+t)q, R(b+t)k⟩: the reason a δ-rotated key attends
    # like a freshly encoded one (Leyline §2.2, Irminsul §2.2)
    rng = np.random.default_rng(9)
    for _ in range(20):
        q, k = rng.standard_normal(64), rng.standard_normal(64)
        a, b, t = (int(v) for v in rng.integers(-50000, 50000, 3))
        s1 = oracle.rotate_f64(q, a, 10000.0) @ oracle.rotate_f64(k, b, 10000.0)
        s2 = oracle.rotate_f64(q, a + t, 10000.0) @ oracle.rotate_f64(k, b + t, 10000.0)
        assert s1 == pytest.approx(s2, abs=1e-8)


def test_pair_norms_are_preserved(oracle):
    # unitary rotation: fp64 exactly up to rounding, bf16 within the rounding of each component
    rng = np.random.default_rng(13)
    for delta in (1, -1008, 32768, -100000):
        x = rng.standard_normal(64)
        y = oracle.rotate_f64(x, delta, 10000.0)
        n0 = np.hypot(x[:32], x[32:])
        assert np.allclose(np.hypot(y[:32], y[32:]), n0, rtol=1e-14)
        xb = synth.bits(torch.from_numpy(x).float().to(torch.bfloat16))
        yb = oracle.rotate_bf16(xb, delta, 10000.0)
        xf, yf = oracle.bf16_to_f64(xb), oracle.bf16_to_f64(yb)
        nb = np.hypot(xf[:32], xf[32:])
        assert np.all(np.abs(np.hypot(yf[:32], yf[32:]) - nb) <= 2.0 ** -8 * nb + 1e-30)


def test_delta_zero_is_the_identity_bitwise(oracle):
    x = np.array([0x8000, 0x0000, 0x3F80, 0x7FC1, 0xFF80, 0x0001] * 8 + [0x4049] * 16,
                 dtype=np.uint16)
    assert np.array_equal(oracle.rotate_bf16(x, 0, 10000.0), x)


def test_bf16_rotation_matches_independent_restatement(oracle):
    rng = np.random.default_rng(17)
    for base, d in ((10000.0, 64), (500000.0, 128)):
        for delta in (1, -1, -1008, 65536, -100000, int(rng.integers(-32768, 32769))):
            xb = synth.bits(synth.bf16_normal((d,), seed=int(rng.integers(1 << 30))))
            assert oracle.rotate_bf16(xb, delta, base).tolist() == ind.rotate_bits(xb, delta, base)


def test_fresh_position_equivalence(oracle):
    # R(δ) applied to a key stored at position i matches the key encoded
    # fresh at i+δ (Leyline §2.2); the two bf16 roundings keep the relative
    # L2 drift under the pages' 4.7e-3 (Leyline §4.3, Irminsul §3).
    rng = np.random.default_rng(19)
    worst = 0.0
    for _ in range(200):
        k = synth.bits(synth.bf16_normal((64,), seed=int(rng.integers(1 << 30))))
        i = int(rng.integers(0, 131072))
        delta = int(rng.integers(-i, 100001))
        stored = oracle.rotate_bf16(k, i, 10000.0)
        moved = oracle.bf16_to_f64(oracle.rotate_bf16(stored, delta, 10000.0))
        fresh = oracle.bf16_to_f64(oracle.rotate_bf16(k, i + delta, 10000.0))
        rel = np.linalg.norm(moved - fresh) / np.linalg.norm(fresh)
        worst = max(worst, rel)
    assert worst <= 4.7e-3


# ---------------------------------------------------------------------------
# Relocation
# ---------------------------------------------------------------------------

def _tiny_pools(seed, L, slots, cd, heads, d, base):
    cp = synth.bits(synth.bf16_normal((L, slots, cd), seed)).copy()
    rt = synth.bits(synth.bf16_normal((L, slots, heads * d), seed + 1)).copy()
    return cp, rt


def _tiny_relocate_case(seed, heads=1, d=8, cd=8, base=10000.0, L=2):
    wl = synth.relocate_workload(seed, num_reqs=3, chunks_per_req=3, len_lo=1, len_hi=9,
                                 delta_lo=-300, delta_hi=300, n_pool_chunks=4, base_hi=11,
                                 block=4)
    sc, sr = _tiny_pools(seed, L, wl.src_slots_total, cd, heads, d, base)
    dc, dr = _tiny_pools(seed + 7, L, wl.dst_slots_total, cd, heads, d, base)
    return wl, sc, sr, dc, dr


@pytest.mark.parametrize("heads,d,cd", [(1, 8, 8), (2, 8, 16), (1, 64, 32)])
def test_relocate_matches_brute_force(oracle, heads, d, cd):
    base = 10000.0
    for seed in range(3):
        wl, sc, sr, dc, dr = _tiny_relocate_case(100 + seed, heads, d, cd, base)
        src = O.Pool(sc, sr, 4, heads, d, base)
        dst = O.Pool(dc.copy(), dr.copy(), 4, heads, d, base)
        st = oracle.relocate(src, dst, wl.tok_off, wl.src_slots, wl.chunk_req, wl.chunk_dst_pos,
                             wl.delta, wl.block_tables)
        assert st == O.OK
        wc, wr = ind.relocate(sc, sr, dc, dr, 4, heads, d, base, wl.tok_off, wl.src_slots,
                              wl.chunk_req, wl.chunk_dst_pos, wl.delta, wl.block_tables)
        assert np.array_equal(dst.copy, wc)
        assert np.array_equal(dst.rot, wr)


def test_relocate_copies_latent_byte_for_byte(oracle):
    # c_KV needs zero correction (Irminsul §2.1; Kamera §2 "byte for byte")
    wl, sc, sr, dc, dr = _tiny_relocate_case(5, 1, 8, 8)
    dst = O.Pool(dc.copy(), dr.copy(), 4, 1, 8, 10000.0)
    assert oracle.relocate(O.Pool(sc, sr, 4, 1, 8, 10000.0), dst, wl.tok_off, wl.src_slots,
                           wl.chunk_req, wl.chunk_dst_pos, wl.delta, wl.block_tables) == O.OK
    for c in range(wl.num_chunks):
        for i in range(int(wl.chunk_len[c])):
            t = int(wl.tok_off[c]) + i
            p = int(wl.chunk_dst_pos[c]) + i
            s = int(wl.block_tables[wl.chunk_req[c], p // 4]) * 4 + p % 4
            assert np.array_equal(dst.copy[:, s], sc[:, wl.src_slots[t]])


def test_relocate_rejects_bad_indices_without_writing(oracle):
    wl, sc, sr, dc, dr = _tiny_relocate_case(6)
    dst = O.Pool(dc.copy(), dr.copy(), 4, 1, 8, 10000.0)
    bad = wl.src_slots.copy()
    bad[-1] = wl.src_slots_total
    assert oracle.relocate(O.Pool(sc, sr, 4, 1, 8, 10000.0), dst, wl.tok_off, bad, wl.chunk_req,
                           wl.chunk_dst_pos, wl.delta, wl.block_tables) == O.ERR_RANGE
    assert np.array_equal(dst.copy, dc) and np.array_equal(dst.rot, dr)


def _patch_factors(wl, L, widths, m, seed, std=0.02):
    T, Cn = wl.total_tokens, wl.num_chunks
    us = [synth.f32_normal((L, T, m), seed + 2 * ch, std=std).numpy() for ch in range(2)]
    vs = [synth.f32_normal((L, Cn, widths[ch], m), seed + 2 * ch + 1, std=std).numpy()
          for ch in range(2)]
    return us, vs


def test_fused_patch_matches_independent_restatement(oracle):
    # KV^ = R(δ)·KV(B|∅) + U_m V_mᵀ with a single rounding (Kamera §2)
    heads, d, cd, m = 2, 8, 16, 3
    wl, sc, sr, dc, dr = _tiny_relocate_case(21, heads, d, cd)
    us, vs = _patch_factors(wl, 2, (cd, heads * d), m, 900, std=0.5)
    dst = O.Pool(dc.copy(), dr.copy(), 4, heads, d, 10000.0)
    pt = O.Patch(m, us, vs)
    assert oracle.relocate(O.Pool(sc, sr, 4, heads, d, 10000.0), dst, wl.tok_off, wl.src_slots,
                           wl.chunk_req, wl.chunk_dst_pos, wl.delta, wl.block_tables, pt) == O.OK
    wc, wr = ind.relocate(sc, sr, dc, dr, 4, heads, d, 10000.0, wl.tok_off, wl.src_slots,
                          wl.chunk_req, wl.chunk_dst_pos, wl.delta, wl.block_tables,
                          patch=(us, vs))
    assert np.array_equal(dst.copy, wc)
    assert np.array_equal(dst.rot, wr)


def _factor_store(wl, seed, widths, m, extra=3, L=2):
    """Factors kept per canonical chunk: a store with more chunks than the
    call, the call's chunks mapped into it in a shuffled order.  Returns the
    store (U, V per channel), the maps and the factors gathered into call
    order (for a call without maps)."""
    rng = np.random.default_rng(seed)
    C = wl.num_chunks
    lens = np.diff(wl.tok_off)
    slots = rng.permutation(C + extra)[:C]                # V slot of each call chunk
    store_len = np.zeros(C + extra, np.int64)
    store_len[slots] = lens
    store_off = np.concatenate([[0], np.cumsum(store_len)[:-1]])
    u_store = [synth.f32_normal((L, int(store_len.sum()) + 5, m), seed + 1 + ch, std=0.4).numpy()
               for ch in range(2)]
    v_store = [synth.f32_normal((L, C + extra, widths[ch], m), seed + 3 + ch, std=0.4).numpy()
               for ch in range(2)]
    u_map = store_off[slots].astype(np.int64)
    rows = np.concatenate([np.arange(u_map[c], u_map[c] + lens[c]) for c in range(C)]
                          ).astype(np.int64)
    u_call = [np.ascontiguousarray(u[:, rows]) for u in u_store]
    v_call = [np.ascontiguousarray(v[:, slots]) for v in v_store]
    return u_store, v_store, u_map, slots.astype(np.int32), u_call, v_call


def test_factor_maps_reuse_factors_kept_per_chunk(oracle):
    # Kamera's reorder / recall: factors stored once per canonical chunk and
    # addressed per call through the maps give what gathering them into call
    # order gives, checked against the independent restatement
    heads, d, cd, m = 2, 8, 16, 4
    wl, sc, sr, dc, dr = _tiny_relocate_case(27, heads, d, cd)
    us, vs, umap, vmap, u_call, v_call = _factor_store(wl, 950, (cd, heads * d), m)
    args = (wl.tok_off, wl.src_slots, wl.chunk_req, wl.chunk_dst_pos, wl.delta, wl.block_tables)
    src = O.Pool(sc, sr, 4, heads, d, 10000.0)
    mapped = O.Pool(dc.copy(), dr.copy(), 4, heads, d, 10000.0)
    assert oracle.relocate(src, mapped, *args, O.Patch(m, us, vs, umap, vmap)) == O.OK
    wc, wr = ind.relocate(sc, sr, dc, dr, 4, heads, d, 10000.0, *args, patch=(u_call, v_call))
    assert np.array_equal(mapped.copy, wc) and np.array_equal(mapped.rot, wr)
    # the standalone patch reads the factors the same way
    a = O.Pool(wc.copy(), wr.copy(), 4, heads, d, 10000.0)
    b = O.Pool(wc.copy(), wr.copy(), 4, heads, d, 10000.0)
    pargs = (wl.tok_off, wl.chunk_req, wl.chunk_dst_pos, wl.block_tables)
    assert oracle.patch_apply(a, *pargs, O.Patch(m, us, vs, umap, vmap)) == O.OK
    assert oracle.patch_apply(b, *pargs, O.Patch(m, u_call, v_call)) == O.OK
    assert np.array_equal(a.copy, b.copy) and np.array_equal(a.rot, b.rot)
    assert not np.array_equal(a.copy, wc)


def test_fused_patch_rounds_once(oracle):
    # a patch fused into the relocation adds to the unrounded rotated value;
    # rounding the rotation first and then the sum differs somewhere
    heads, d, cd, m = 1, 64, 8, 4
    wl, sc, sr, dc, dr = _tiny_relocate_case(23, heads, d, cd)
    us, vs = _patch_factors(wl, 2, (cd, d), m, 40, std=0.3)
    us[0] = vs[0] = None
    fused = O.Pool(dc.copy(), dr.copy(), 4, heads, d, 10000.0)
    src = O.Pool(sc, sr, 4, heads, d, 10000.0)
    args = (wl.tok_off, wl.src_slots, wl.chunk_req, wl.chunk_dst_pos, wl.delta, wl.block_tables)
    assert oracle.relocate(src, fused, *args, O.Patch(m, us, vs)) == O.OK
    twice = O.Pool(dc.copy(), dr.copy(), 4, heads, d, 10000.0)
    assert oracle.relocate(src, twice, *args) == O.OK
    assert oracle.patch_apply(twice, wl.tok_off, wl.chunk_req, wl.chunk_dst_pos, wl.block_tables,
                              O.Patch(m, us, vs)) == O.OK
    rotated = O.Pool(dc.copy(), dr.copy(), 4, heads, d, 10000.0)
    assert oracle.relocate(src, rotated, *args) == O.OK
    diff = oracle.bf16_to_f64(fused.rot) - oracle.bf16_to_f64(twice.rot)
    assert np.any(diff != 0)
    # the two-step path adds one extra rounding at the scale of the rotated
    # value: |diff| <= ulp(rotated)/2 + ulp(result), ulp(v) <= 2^-7 |v|
    bound = (2.0 ** -8 * np.abs(oracle.bf16_to_f64(rotated.rot))
             + 2.0 ** -7 * np.abs(oracle.bf16_to_f64(fused.rot)))
    assert np.all(np.abs(diff) <= bound * 1.001 + 1e-30)


def test_rank_one_one_hot_patch_touches_one_value(oracle):
    heads, d, cd, m = 1, 8, 8, 1
    wl, sc, sr, dc, dr = _tiny_relocate_case(25, heads, d, cd)
    pool = O.Pool(dc.copy(), dr.copy(), 4, heads, d, 10000.0)
    L, T, Cn = 2, wl.total_tokens, wl.num_chunks
    u = np.zeros((L, T, m), np.float32)
    v = np.zeros((L, Cn, cd, m), np.float32)
    c0 = Cn - 1
    t0 = int(wl.tok_off[c0]) + int(wl.chunk_len[c0]) - 1
    col0, l0 = 5, 1
    u[l0, t0, 0] = 0.75
    v[l0, c0, col0, 0] = 1.5
    assert oracle.patch_apply(pool, wl.tok_off, wl.chunk_req, wl.chunk_dst_pos, wl.block_tables,
                              O.Patch(m, [u, None], [v, None])) == O.OK
    p = int(wl.chunk_dst_pos[c0]) + int(wl.chunk_len[c0]) - 1
    s = int(wl.block_tables[wl.chunk_req[c0], p // 4]) * 4 + p % 4
    changed = np.argwhere(pool.copy != dc)
    x = float(oracle.bf16_to_f64(dc[l0, s, col0]))
    want = ind.round_bf16(x + 0.75 * 1.5)
    if want == dc[l0, s, col0]:
        assert len(changed) == 0
    else:
        assert changed.tolist() == [[l0, s, col0]]
        assert pool.copy[l0, s, col0] == want
    assert np.array_equal(pool.rot, dr)


def test_standalone_patch_matches_numpy_matmul(oracle):
    heads, d, cd, m = 2, 8, 16, 5
    wl, sc, sr, dc, dr = _tiny_relocate_case(27, heads, d, cd)
    us, vs = _patch_factors(wl, 2, (cd, heads * d), m, 77, std=0.4)
    pool = O.Pool(dc.copy(), dr.copy(), 4, heads, d, 10000.0)
    assert oracle.patch_apply(pool, wl.tok_off, wl.chunk_req, wl.chunk_dst_pos, wl.block_tables,
                              O.Patch(m, us, vs)) == O.OK
    for ch, (orig, got) in enumerate(((dc, pool.copy), (dr, pool.rot))):
        want = orig.copy()
        for c in range(wl.num_chunks):
            for i in range(int(wl.chunk_len[c])):
                t = int(wl.tok_off[c]) + i
                p = int(wl.chunk_dst_pos[c]) + i
                s = int(wl.block_tables[wl.chunk_req[c], p // 4]) * 4 + p % 4
                for l in range(2):
                    add = us[ch][l, t].astype(np.float64) @ vs[ch][l, c].astype(np.float64).T
                    x = oracle.bf16_to_f64(orig[l, s])
                    want[l, s] = [ind.round_bf16(float(a)) for a in x + add]
        assert np.array_equal(got, want)


# ---------------------------------------------------------------------------
# Splice
# ---------------------------------------------------------------------------

def test_delta_of_the_single_layer_directive():
    # Leyline §2.2: Δ = |R| - |S|.  The 4096-token single-layer workload
    # replaces [1024, 2048) by a 16-row stub.
    s_start, s_end, n_r, n = 1024, 2048, 16, 4096
    delta = n_r - (s_end - s_start)
    assert delta == -1008
    assert n + delta == 3088
    assert (s_end + delta) == s_start + n_r      # first downstream row lands right after the stub


def _splice_pool(seed, seq_lens, max_blocks, heads=1, d=8, cd=8, L=2, block=4, spare=2):
    ss = synth.splice_seqs(seed, seq_lens, max_blocks, block=block, spare_blocks=spare)
    cp, rt = _tiny_pools(seed, L, ss.num_slots, cd, heads, d, 10000.0)
    return ss, cp, rt


def test_splice_brute_force_every_directive(oracle):
    # every (s_start, s_end, |R|) on a 12-token cache with 4-token blocks,
    # Δ of both signs (Leyline §2.1-§2.3), against list slicing
    n, maxb, L, heads, d, cd = 12, 6, 2, 1, 8, 8
    ss, cp, rt = _splice_pool(31, [n], maxb, heads, d, cd, L)
    stub_c = synth.bits(synth.bf16_normal((L, 8, cd), 32)).copy()
    stub_r = synth.bits(synth.bf16_normal((L, 8, heads * d), 33)).copy()
    cases = 0
    for a in range(n + 1):
        for b in range(a, n + 1):
            for nr in range(0, 9):
                if n + nr - (b - a) > maxb * 4:
                    continue
                pool = O.Pool(cp.copy(), rt.copy(), 4, heads, d, 10000.0)
                lens = np.array([n], np.int32)
                sc = np.ascontiguousarray(stub_c[:, :nr])
                sr = np.ascontiguousarray(stub_r[:, :nr])
                st = oracle.splice(pool, ss.block_tables, lens, [a], [b], [nr], sc, sr)
                assert st == O.OK
                wc, wr, wl = ind.splice(cp, rt, 4, heads, d, 10000.0, ss.block_tables, [n], [a],
                                        [b], [nr], sc, sr)
                assert lens.tolist() == wl
                assert np.array_equal(pool.copy, wc) and np.array_equal(pool.rot, wr)
                cases += 1
    assert cases > 700


def test_splice_batch_of_sequences_with_gqa_heads(oracle):
    lens = [13, 0, 29, 7]
    ss, cp, rt = _splice_pool(41, lens, 10, heads=2, d=8, cd=16)
    dirs = synth.random_directives(42, lens, 0, 12, 0, 9)
    tot = int(dirs.stub_len.sum())
    sc = synth.bits(synth.bf16_normal((2, tot, 16), 43)).copy()
    sr = synth.bits(synth.bf16_normal((2, tot, 16), 44)).copy()
    pool = O.Pool(cp.copy(), rt.copy(), 4, 2, 8, 10000.0)
    seq = np.array(lens, np.int32)
    assert oracle.splice(pool, ss.block_tables, seq, dirs.s_start, dirs.s_end, dirs.stub_len, sc,
                         sr) == O.OK
    wc, wr, wl = ind.splice(cp, rt, 4, 2, 8, 10000.0, ss.block_tables, lens, dirs.s_start,
                            dirs.s_end, dirs.stub_len, sc, sr)
    assert seq.tolist() == wl
    assert np.array_equal(pool.copy, wc) and np.array_equal(pool.rot, wr)


def test_splice_leaves_unreferenced_blocks_alone(oracle):
    ss, cp, rt = _splice_pool(51, [10, 11], 6, spare=3)
    pool = O.Pool(cp.copy(), rt.copy(), 4, 1, 8, 10000.0)
    sc = synth.bits(synth.bf16_normal((2, 9, 8), 52)).copy()
    sr = synth.bits(synth.bf16_normal((2, 9, 8), 53)).copy()
    seq = np.array([10, 11], np.int32)
    assert oracle.splice(pool, ss.block_tables, seq, [2, 0], [3, 11], [5, 4], sc, sr) == O.OK
    used = set(ss.block_tables.ravel().tolist())
    for blk in range(ss.num_slots // 4):
        if blk not in used:
            sl = slice(blk * 4, blk * 4 + 4)
            assert np.array_equal(pool.copy[:, sl], cp[:, sl])


def test_splice_delta_zero_only_overwrites_the_span(oracle):
    ss, cp, rt = _splice_pool(61, [12], 4)
    pool = O.Pool(cp.copy(), rt.copy(), 4, 1, 8, 10000.0)
    sc = synth.bits(synth.bf16_normal((2, 3, 8), 62)).copy()
    sr = synth.bits(synth.bf16_normal((2, 3, 8), 63)).copy()
    seq = np.array([12], np.int32)
    assert oracle.splice(pool, ss.block_tables, seq, [4], [7], [3], sc, sr) == O.OK
    assert seq.tolist() == [12]
    for p in range(12):
        s = int(ss.block_tables[0, p // 4]) * 4 + p % 4
        if 4 <= p < 7:
            assert np.array_equal(pool.copy[:, s], sc[:, p - 4])
            assert np.array_equal(pool.rot[:, s], sr[:, p - 4])
        else:
            assert np.array_equal(pool.copy[:, s], cp[:, s])
            assert np.array_equal(pool.rot[:, s], rt[:, s])


def test_splice_forget_truncates_without_moving_data(oracle):
    ss, cp, rt = _splice_pool(71, [12, 9], 5)
    pool = O.Pool(cp.copy(), rt.copy(), 4, 1, 8, 10000.0)
    seq = np.array([12, 9], np.int32)
    assert oracle.splice(pool, ss.block_tables, seq, [3, 0], [5, 9], [2, 1], None, None,
                         O.FORGET) == O.OK
    assert seq.tolist() == [3, 0]
    assert np.array_equal(pool.copy, cp) and np.array_equal(pool.rot, rt)


def test_splice_argument_errors(oracle):
    ss, cp, rt = _splice_pool(81, [12], 3)
    pool = O.Pool(cp.copy(), rt.copy(), 4, 1, 8, 10000.0)
    sc = np.zeros((2, 8, 8), np.uint16)
    seq = np.array([12], np.int32)
    assert oracle.splice(pool, ss.block_tables, seq, [5], [4], [0], sc, sc) == O.ERR_INVALID
    assert oracle.splice(pool, ss.block_tables, seq, [5], [13], [0], sc, sc) == O.ERR_INVALID
    assert oracle.splice(pool, ss.block_tables, seq, [5], [6], [2], sc, sc) == O.ERR_CAPACITY
    assert seq.tolist() == [12] and np.array_equal(pool.copy, cp)


def test_successive_directives_round_between_calls(oracle):
    # directives are applied one after another on the stored (bf16) cache
    ss, cp, rt = _splice_pool(91, [12], 6)
    sc = synth.bits(synth.bf16_normal((2, 4, 8), 92)).copy()
    sr = synth.bits(synth.bf16_normal((2, 4, 8), 93)).copy()
    pool = O.Pool(cp.copy(), rt.copy(), 4, 1, 8, 10000.0)
    seq = np.array([12], np.int32)
    c, r, lens = cp, rt, [12]
    for a, b, nr in ((1, 4, 2), (6, 7, 4), (0, 2, 1)):
        sub_c, sub_r = np.ascontiguousarray(sc[:, :nr]), np.ascontiguousarray(sr[:, :nr])
        assert oracle.splice(pool, ss.block_tables, seq, [a], [b], [nr], sub_c, sub_r) == O.OK
        c, r, lens = ind.splice(c, r, 4, 1, 8, 10000.0, ss.block_tables, lens, [a], [b], [nr],
                                sub_c, sub_r)
    assert seq.tolist() == lens
    assert np.array_equal(pool.copy, c) and np.array_equal(pool.rot, r)


# ---------------------------------------------------------------------------
# Composed directives: every row moved once, rotated by its total shift,
# rounded once (Leyline §2.2-§2.3 with R(a)R(b) = R(a+b))
# ---------------------------------------------------------------------------

def _stubs(seed, L, n, cd, rw):
    sc = synth.bits(synth.bf16_normal((L, max(n, 1), cd), seed)).copy()
    sr = synth.bits(synth.bf16_normal((L, max(n, 1), rw), seed + 1)).copy()
    return np.ascontiguousarray(sc[:, :n]), np.ascontiguousarray(sr[:, :n])


def _random_dirs(rng, lens, k, max_span, max_stub, cap):
    """k directives per sequence, each valid in the indexing the previous left."""
    cur = list(lens)
    dirs = []
    for _ in range(k):
        a_s, b_s, n_s = [], [], []
        for q, n in enumerate(cur):
            a = int(rng.integers(0, n + 1))
            b = int(rng.integers(a, min(n, a + max_span) + 1))
            nr = int(rng.integers(0, max_stub + 1))
            nr = min(nr, cap - (n - (b - a)))
            a_s.append(a)
            b_s.append(b)
            n_s.append(nr)
            cur[q] = n + nr - (b - a)
        dirs.append((a_s, b_s, n_s))
    return dirs


def _dir_arrays(dirs):
    return tuple(np.asarray([d[j] for d in dirs], np.int32) for j in range(3))


def test_composed_single_directive_is_the_splice(oracle):
    # with one directive the composed edit is the plain splice, bit for bit
    rng = np.random.default_rng(101)
    for seed, heads, d, cd in ((102, 1, 8, 8), (103, 2, 8, 16)):
        lens = [13, 0, 21, 9]
        ss, cp, rt = _splice_pool(seed, lens, 9, heads, d, cd)
        dirs = _random_dirs(rng, lens, 1, 10, 8, 9 * 4)
        s0, s1, nr = _dir_arrays(dirs)
        sc, sr = _stubs(seed + 5, 2, int(nr.sum()), cd, heads * d)
        p1 = O.Pool(cp.copy(), rt.copy(), 4, heads, d, 10000.0)
        p2 = O.Pool(cp.copy(), rt.copy(), 4, heads, d, 10000.0)
        l1, l2 = np.array(lens, np.int32), np.array(lens, np.int32)
        assert oracle.splice(p1, ss.block_tables, l1, s0[0], s1[0], nr[0], sc, sr) == O.OK
        assert oracle.splice_composed(p2, ss.block_tables, l2, s0, s1, nr, sc, sr) == O.OK
        assert l1.tolist() == l2.tolist()
        assert np.array_equal(p1.copy, p2.copy) and np.array_equal(p1.rot, p2.rot)


def test_composed_brute_force_two_directives(oracle):
    # many directive pairs on a 10-token cache, against symbolic list slicing
    # with one complex rotation per row
    n, maxb = 10, 7
    ss, cp, rt = _splice_pool(111, [n], maxb)
    rng = np.random.default_rng(112)
    cases = 0
    for _ in range(160):
        dirs = _random_dirs(rng, [n], 2, 6, 6, maxb * 4)
        s0, s1, nr = _dir_arrays(dirs)
        sc, sr = _stubs(113, 2, int(nr.sum()), 8, 8)
        pool = O.Pool(cp.copy(), rt.copy(), 4, 1, 8, 10000.0)
        lens = np.array([n], np.int32)
        assert oracle.splice_composed(pool, ss.block_tables, lens, s0, s1, nr, sc, sr) == O.OK
        wc, wr, wl = ind.splice_composed(cp, rt, 4, 1, 8, 10000.0, ss.block_tables, [n], dirs,
                                         sc, sr)
        assert lens.tolist() == wl
        assert np.array_equal(pool.copy, wc) and np.array_equal(pool.rot, wr)
        cases += 1
    assert cases == 160


def test_composed_three_directives_batch_gqa(oracle):
    lens = [17, 5, 0, 26]
    ss, cp, rt = _splice_pool(121, lens, 12, heads=2, d=8, cd=16)
    dirs = _random_dirs(np.random.default_rng(122), lens, 3, 9, 7, 12 * 4)
    s0, s1, nr = _dir_arrays(dirs)
    sc, sr = _stubs(123, 2, int(nr.sum()), 16, 16)
    pool = O.Pool(cp.copy(), rt.copy(), 4, 2, 8, 10000.0)
    seq = np.array(lens, np.int32)
    assert oracle.splice_composed(pool, ss.block_tables, seq, s0, s1, nr, sc, sr) == O.OK
    wc, wr, wl = ind.splice_composed(cp, rt, 4, 2, 8, 10000.0, ss.block_tables, lens, dirs, sc, sr)
    assert seq.tolist() == wl
    assert np.array_equal(pool.copy, wc) and np.array_equal(pool.rot, wr)


def test_composed_differs_from_successive_calls_only_where_rows_rounded_twice(oracle):
    # rows shifted by at most one of the directives are rotated once either
    # way and agree bit for bit; rows shifted more than once are rounded once
    # here and once per shift by successive calls
    n = 40
    ss, cp, rt = _splice_pool(131, [n], 16, d=16)
    dirs = [([3], [9], [2]), ([20], [20], [5]), ([30], [34], [0])]
    s0, s1, nr = _dir_arrays(dirs)
    sc, sr = _stubs(132, 2, int(nr.sum()), 8, 16)
    comp = O.Pool(cp.copy(), rt.copy(), 4, 1, 16, 10000.0)
    lc = np.array([n], np.int32)
    assert oracle.splice_composed(comp, ss.block_tables, lc, s0, s1, nr, sc, sr) == O.OK
    succ = O.Pool(cp.copy(), rt.copy(), 4, 1, 16, 10000.0)
    ls = np.array([n], np.int32)
    off = 0
    for a, b, k in dirs:
        assert oracle.splice(succ, ss.block_tables, ls, a, b, k, np.ascontiguousarray(
            sc[:, off:off + k[0]]), np.ascontiguousarray(sr[:, off:off + k[0]])) == O.OK
        off += k[0]
    assert lc.tolist() == ls.tolist() == [n + 2 - 6 + 5 - 4]
    # shifts seen by each final position: track the edits symbolically
    seq = [[0, 0] for _ in range(n)]                   # [nonzero shifts, 0]
    for a, b, k in dirs:
        delta = k[0] - (b[0] - a[0])
        seq = seq[:a[0]] + [[0, 0] for _ in range(k[0])] + [
            [c + (delta != 0), 0] for c, _ in seq[b[0]:]]
    once = twice = 0
    for p, (shifts, _) in enumerate(seq):
        s = int(ss.block_tables[0, p // 4]) * 4 + p % 4
        assert np.array_equal(comp.copy[:, s], succ.copy[:, s])
        if shifts <= 1:
            assert np.array_equal(comp.rot[:, s], succ.rot[:, s]), p
            once += 1
        else:
            twice += 1
    assert once > 0 and twice > 0


def test_composed_insert_then_remove_restores_the_cache(oracle):
    # insert 7 stub rows at 5, then remove exactly them: every row's total
    # shift is 0, so the cache comes back bit for bit
    n = 23
    ss, cp, rt = _splice_pool(141, [n], 10)
    sc, sr = _stubs(142, 2, 7, 8, 8)
    pool = O.Pool(cp.copy(), rt.copy(), 4, 1, 8, 10000.0)
    seq = np.array([n], np.int32)
    s0, s1, nr = _dir_arrays([([5], [5], [7]), ([5], [12], [0])])
    assert oracle.splice_composed(pool, ss.block_tables, seq, s0, s1, nr, sc, sr) == O.OK
    assert seq.tolist() == [n]
    assert np.array_equal(pool.copy, cp) and np.array_equal(pool.rot, rt)


def test_composed_checks_final_capacity_and_each_directive(oracle):
    ss, cp, rt = _splice_pool(151, [12], 4)              # capacity 16 tokens
    sc, sr = _stubs(152, 2, 12, 8, 8)
    pool = O.Pool(cp.copy(), rt.copy(), 4, 1, 8, 10000.0)
    # grows to 22 in between, ends at 12: only the final length counts
    s0, s1, nr = _dir_arrays([([0], [0], [10]), ([0], [10], [0])])
    seq = np.array([12], np.int32)
    assert oracle.splice_composed(pool, ss.block_tables, seq, s0, s1, nr, sc, sr) == O.OK
    assert seq.tolist() == [12]
    # ends at 18 > 16
    s0, s1, nr = _dir_arrays([([0], [0], [10]), ([0], [4], [0])])
    seq = np.array([12], np.int32)
    assert oracle.splice_composed(pool, ss.block_tables, seq, s0, s1, nr, sc, sr) == O.ERR_CAPACITY
    assert seq.tolist() == [12]
    # the second directive's span lies beyond the length the first one left
    before_c, before_r = pool.copy.copy(), pool.rot.copy()
    s0, s1, nr = _dir_arrays([([2], [10], [0]), ([3], [5], [1])])
    seq = np.array([12], np.int32)
    assert oracle.splice_composed(pool, ss.block_tables, seq, s0, s1, nr, sc, sr) == O.ERR_INVALID
    assert seq.tolist() == [12]
    assert np.array_equal(pool.copy, before_c) and np.array_equal(pool.rot, before_r)


# ---------------------------------------------------------------------------
# Interleaved pairing: pair j = (x[2j], x[2j+1]), same θ_j
# ---------------------------------------------------------------------------

@pytest.mark.parametrize("d", [8, 64, 128])
def test_interleaved_rotation_is_complex_multiplication(oracle, d):
    rng = np.random.default_rng(160 + d)
    x = synth.bits(synth.bf16_normal((d,), 161 + d)).copy()
    for delta in (1, -7, 999, 65536, -100000):
        got = oracle.rotate_bf16(x, delta, 10000.0, interleaved=True)
        assert got.tolist() == ind.rotate_bits(x, delta, 10000.0, il=True), delta
    assert oracle.rotate_bf16(x, 0, 10000.0, interleaved=True).tolist() == x.tolist()
    del rng


def test_interleaved_is_rotate_half_under_the_index_permutation(oracle):
    # moving x[2j] -> j and x[2j+1] -> j + d/2 turns one pairing into the other
    d = 64
    perm = np.concatenate([np.arange(0, d, 2), np.arange(1, d, 2)])
    for seed in range(4):
        x = synth.bits(synth.bf16_normal((d,), 170 + seed)).copy()
        for delta in (3, -4096, 77777):
            il = oracle.rotate_bf16(x, delta, 500000.0, interleaved=True)
            half = oracle.rotate_bf16(x[perm], delta, 500000.0)
            back = np.empty_like(half)
            back[perm] = half
            assert np.array_equal(il, back)
            assert not np.array_equal(il, oracle.rotate_bf16(x, delta, 500000.0))


def test_interleaved_relocate_and_splice_match_the_restatement(oracle):
    heads, d, cd = 2, 8, 8
    wl, sc, sr, dc, dr = _tiny_relocate_case(181, heads, d, cd)
    src = O.Pool(sc, sr, 4, heads, d, 10000.0, pair_convention=1)
    dst = O.Pool(dc.copy(), dr.copy(), 4, heads, d, 10000.0, pair_convention=1)
    args = (wl.tok_off, wl.src_slots, wl.chunk_req, wl.chunk_dst_pos, wl.delta, wl.block_tables)
    assert oracle.relocate(src, dst, *args) == O.OK
    wc, wr = ind.relocate(sc, sr, dc, dr, 4, heads, d, 10000.0, *args, il=True)
    assert np.array_equal(dst.copy, wc) and np.array_equal(dst.rot, wr)
    # conventions must agree between the pools
    mixed = O.Pool(dc.copy(), dr.copy(), 4, heads, d, 10000.0)
    assert oracle.relocate(src, mixed, *args) == O.ERR_INVALID
    lens = [13, 21]
    ss, cp, rt = _splice_pool(182, lens, 9, heads, d, cd)
    d0 = synth.random_directives(183, np.asarray(lens, np.int32), 0, 10, 0, 7)
    tot = int(d0.stub_len.sum())
    stc = synth.bits(synth.bf16_normal((2, max(tot, 1), cd), 184)).copy()[:, :tot]
    str_ = synth.bits(synth.bf16_normal((2, max(tot, 1), heads * d), 185)).copy()[:, :tot]
    stc, str_ = np.ascontiguousarray(stc), np.ascontiguousarray(str_)
    pool = O.Pool(cp.copy(), rt.copy(), 4, heads, d, 10000.0, pair_convention=1)
    seq = np.array(lens, np.int32)
    assert oracle.splice(pool, ss.block_tables, seq, d0.s_start, d0.s_end, d0.stub_len, stc,
                         str_) == O.OK
    wc, wr, wl2 = ind.splice(cp, rt, 4, heads, d, 10000.0, ss.block_tables, lens, d0.s_start,
                             d0.s_end, d0.stub_len, stc, str_, il=True)
    assert seq.tolist() == wl2
    assert np.array_equal(pool.copy, wc) and np.array_equal(pool.rot, wr)


def test_mla_row_split():
    # Irminsul §2.1: cKV is 89% of the MLA row, k_r 11%
    assert round(512 / 576 * 100) == 89 and round(64 / 576 * 100) == 11
    assert (512 + 64) * 2 == 1152
