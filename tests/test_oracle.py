"""Pins for the CPU oracle: each test checks the oracle against something other
than itself - the format's code table, an independent library conversion
(torch's float8_e4m3fn), brute force over exact rationals, hand-worked blocks,
closed forms and invariants. No GPU is involved."""
from fractions import Fraction
from pathlib import Path

import numpy as np
import pytest
import torch

import oracle as O

GOLDEN = Path(__file__).parent / "golden"
F32 = np.float32

# The format's fixed code table (magnitudes of codes 0..7; bit 3 is the sign).
E2M1_TABLE = [0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0]


def load_blocks():
    blocks, cur = [], None
    for line in (GOLDEN / "quantize_blocks.txt").read_text().splitlines():
        line = line.strip()
        if not line or line.startswith("#"):
            continue
        key, _, rest = line.partition(" ")
        if key == "block":
            cur = {"name": rest}
            blocks.append(cur)
        elif key == "s_t":
            cur["s_t"] = float(rest)
        elif key == "x":
            cur["x"] = [float(v) for v in rest.split()]
        elif key == "scale":
            cur["scale"] = int(rest, 16)
        elif key == "codes":
            cur["codes"] = [int(v, 16) for v in rest.split()]
        elif key == "packed":
            cur["packed"] = [int(v, 16) for v in rest.split()]
    return blocks


# ----------------------------------------------------------------- e2m1 codec

def test_e2m1_decode_is_the_code_table():
    vals = O.e2m1_value(np.arange(16))
    assert list(vals[:8]) == E2M1_TABLE
    assert list(vals[8:]) == [-v for v in E2M1_TABLE]
    assert np.signbit(vals[8])          # code 0x8 is negative zero


def _brute_e2m1(x: float) -> int:
    """Nearest magnitude by exact rational distance; ties to the even code."""
    fx = Fraction(x)
    mag = abs(fx)
    best = None
    for code, v in enumerate(E2M1_TABLE):
        d = abs(mag - Fraction(v))
        if best is None or d < best[0] or (d == best[0] and code % 2 == 0):
            best = (d, code)
    code = best[1]
    if mag > 6:
        code = 7
    return code | (8 if np.signbit(x) else 0)


def test_e2m1_encode_brute_force():
    grid = list(np.arange(-8, 8, 1 / 128, dtype=np.float64))
    mids = [0.25, 0.75, 1.25, 1.75, 2.5, 3.5, 5.0]
    for m in mids:
        for s in (1.0, -1.0):
            v = F32(s * m)
            grid += [float(v), float(np.nextafter(v, F32(np.inf))), float(np.nextafter(v, F32(-np.inf)))]
    grid += [0.0, -0.0, 1e-30, -1e-30, 6.0, 6.5, 1e9, -1e9]
    xs = np.array(grid, dtype=np.float32)
    got = O.e2m1_encode(xs)
    want = np.array([_brute_e2m1(float(x)) for x in xs], dtype=np.uint8)
    np.testing.assert_array_equal(got, want)


def test_e2m1_encode_ties_and_signed_zero():
    # (a list, not a dict: 0.0 and -0.0 compare equal as keys)
    cases = [(0.25, 0x0), (0.75, 0x2), (1.25, 0x2), (1.75, 0x4), (2.5, 0x4), (3.5, 0x6),
             (5.0, 0x6), (7.0, 0x7), (-0.25, 0x8), (-0.0, 0x8), (0.0, 0x0), (-0.1, 0x8), (-5.0, 0xE)]
    xs = np.array([c[0] for c in cases], dtype=np.float32)
    assert list(O.e2m1_encode(xs)) == [c[1] for c in cases]
    assert O.e2m1_encode(np.array([np.inf], np.float32))[0] == 7


# ----------------------------------------------------------------- E4M3 codec

def test_e4m3_decode_matches_torch_float8():
    codes = torch.arange(256, dtype=torch.int32).to(torch.uint8)
    ref = codes.view(torch.float8_e4m3fn).to(torch.float64).numpy()
    got = O.e4m3_value(np.arange(256))
    np.testing.assert_array_equal(np.isnan(got), np.isnan(ref))
    ok = ~np.isnan(ref)
    np.testing.assert_array_equal(got[ok], ref[ok])
    assert np.isnan(got).sum() == 2   # 0x7F and 0xFF


def test_e4m3_known_values():
    v = O.e4m3_value(np.array([0x7E, 0x01, 0x07, 0x08, 0x38, 0x15, 0x80]))
    assert list(v) == [448.0, 2.0 ** -9, 7 * 2.0 ** -9, 2.0 ** -6, 1.0, 0.05078125, -0.0]


def test_e4m3_encode_roundtrip_all_codes():
    codes = np.arange(0x7F)
    np.testing.assert_array_equal(O.e4m3_encode(O.e4m3_value(codes).astype(np.float32)), codes)


def test_e4m3_encode_matches_torch_in_range():
    rng = np.random.default_rng(1)
    vals = O.e4m3_value(np.arange(0x7F))
    mids = (vals[1:] + vals[:-1]) / 2
    xs = [rng.uniform(0, 460, 200_000).astype(np.float32),
          np.exp2(rng.uniform(-14, 8.8, 200_000)).astype(np.float32)]
    for m in mids.astype(np.float32):
        xs.append(np.array([m, np.nextafter(m, F32(np.inf)), np.nextafter(m, F32(0))], np.float32))
    x = np.concatenate(xs)
    x = x[x <= 460]
    ref = torch.from_numpy(x).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    np.testing.assert_array_equal(O.e4m3_encode(x), ref)


def test_e4m3_encode_saturates_and_rounds_tiny_to_zero():
    x = np.array([448.0, 470.0, 1e6, np.inf, 2.0 ** -10, 2.0 ** -10 * 1.0001, 0.0], np.float32)
    assert list(O.e4m3_encode(x)) == [0x7E, 0x7E, 0x7E, 0x7E, 0x00, 0x01, 0x00]


# ---------------------------------------------------------- hand-worked blocks

@pytest.mark.parametrize("blk", load_blocks(), ids=lambda b: "block" + b["name"])
def test_golden_block(blk):
    x = np.array([blk["x"]], dtype=np.float32)
    # every fixture value is exact in bf16, so the bf16 path sees the same x
    assert np.array_equal(torch.from_numpy(x).to(torch.bfloat16).float().numpy(), x)
    qt = O.quantize(x, s_t=blk["s_t"])
    assert qt.scales[0, 0] == blk["scale"]
    assert list(O.unpack_codes(qt.codes)[0]) == blk["codes"]
    assert list(qt.codes[0]) == blk["packed"]


def test_golden_block1_decodes_to_rounded_values():
    blk = load_blocks()[0]
    qt = O.quantize(np.array([blk["x"]], np.float32), s_t=1.0)
    want = [0, 0, 0, .5, 1, 1, 2, 2, 4, 4, 6, -0.0, -1, -3, -6, -0.0]
    got = O.decode(qt)[0]
    assert list(got) == want
    assert list(np.signbit(got)) == list(np.signbit(np.array(want)))


# ------------------------------------------------------------- tensor scale

def test_tensor_scale_closed_form():
    x = torch.randn(64, 512, generator=torch.Generator().manual_seed(3)) * 7
    x_np = x.numpy()
    want = (x.abs().amax() / torch.tensor(2688.0, dtype=torch.float32)).item()
    assert O.tensor_scale(x_np) == F32(want)
    assert O.quantize(x_np).s_t == F32(want)
    assert O.tensor_scale(np.zeros((2, 16), np.float32)) == 1.0


def test_largest_block_gets_scale_448_when_dynamic():
    rng = np.random.default_rng(2)
    x = rng.standard_normal((32, 256)).astype(np.float32)
    qt = O.quantize(x)
    # the block holding the tensor amax has sb = amax / (6 * amax / 2688) ~ 448
    r, c = np.unravel_index(np.argmax(np.abs(x)), x.shape)
    assert qt.scales[r, c // 16] == 0x7E


# ---------------------------------------------------------------- invariants

def test_roundtrip_requantize_is_identity():
    rng = np.random.default_rng(4)
    R, K = 64, 256
    codes = rng.integers(0, 16, (R, K)).astype(np.uint8)
    # every block holds a +-6 so its amax is exactly 6 * scale
    codes[:, ::16] = rng.choice([0x7, 0xF], size=(R, K // 16))
    scales = rng.integers(1, 0x7F, (R, K // 16)).astype(np.uint8)
    qt = O.QTensor(O.pack_codes(codes), scales, 1.0)
    x = O.decode(qt).astype(np.float32)
    back = O.quantize(x, s_t=1.0)
    np.testing.assert_array_equal(back.scales, scales)
    np.testing.assert_array_equal(back.codes, qt.codes)


def test_sign_symmetry():
    rng = np.random.default_rng(5)
    x = (rng.standard_normal((16, 128)) * 0.02).astype(np.float32)
    a, b = O.quantize(x), O.quantize(-x)
    np.testing.assert_array_equal(a.scales, b.scales)
    np.testing.assert_array_equal(a.codes ^ 0x88, b.codes)


def test_power_of_two_shift_moves_only_the_scale():
    rng = np.random.default_rng(6)
    x = rng.uniform(0.5, 1.0, (8, 64)).astype(np.float32) * rng.choice([-1, 1], (8, 64))
    base = O.quantize(x, s_t=1.0)
    e = (base.scales >> 3) & 0xF
    assert e.min() >= 2 and e.max() <= 10
    for j in (-1, 1, 3):
        sh = O.quantize((x * F32(2.0 ** j)).astype(np.float32), s_t=1.0)
        np.testing.assert_array_equal(sh.codes, base.codes)
        np.testing.assert_array_equal(sh.scales.astype(int), base.scales.astype(int) + 8 * j)


def test_error_is_at_most_half_a_gap():
    rng = np.random.default_rng(7)
    x = torch.from_numpy(rng.standard_t(4, (64, 512)).astype(np.float32)).to(torch.bfloat16).float().numpy()
    qt = O.quantize(x)
    xh = O.decode(qt)
    codes = O.unpack_codes(qt.codes) & 7
    den = np.repeat(O.e4m3_value(qt.scales), 16, axis=1) * np.float64(qt.s_t)
    gaps = np.array([0.5, 0.5, 0.5, 0.5, 1.0, 1.0, 2.0, 2.0])      # gap to the neighbour
    bound = 0.5 * gaps[codes] * den * (1 + 2.0 ** -20)
    sat = (codes == 7) & (np.abs(x) > 6 * den)
    assert np.all((np.abs(x - xh) <= bound) | sat)
    # saturation is reachable only by the small excess the rounded scale allows
    assert np.all(np.abs(x)[sat] <= 6 * den[sat] * (1 + 2.0 ** -4) * (1 + 2.0 ** -20))


# --------------------------------------------------------------------- GEMMs

def _brute_gemm(x, qt):
    """Exact rational GEMM from the code table literal and E4M3 bit fields."""
    codes = O.unpack_codes(qt.codes)
    N, K = codes.shape
    M = len(x)
    st = Fraction(float(qt.s_t))
    out = [[Fraction(0)] * N for _ in range(M)]
    for n in range(N):
        w = []
        for k in range(K):
            c = int(codes[n, k])
            v = Fraction(E2M1_TABLE[c & 7]) * (-1 if c & 8 else 1)
            s = int(qt.scales[n, k // 16])
            e, m = (s >> 3) & 0xF, s & 7
            sv = Fraction(m, 8) * Fraction(1, 64) if e == 0 else (1 + Fraction(m, 8)) * Fraction(2) ** (e - 7)
            w.append(v * sv * st)
        for i in range(M):
            out[i][n] = sum(Fraction(float(x[i][k])) * w[k] for k in range(K))
    return out


@pytest.mark.parametrize("M,N,K", [(1, 1, 16), (2, 3, 32), (3, 17, 48), (1, 5, 16)])
def test_gemm_w4a16_brute_force(M, N, K):
    rng = np.random.default_rng(M * 100 + N * 10 + K)
    w = (rng.standard_normal((N, K)) * 0.02).astype(np.float32)
    x = torch.from_numpy(rng.standard_normal((M, K)).astype(np.float32)).to(torch.bfloat16).float().numpy()
    qt = O.quantize(w)
    got = O.gemm_w4a16(x, qt)
    want = _brute_gemm(x, qt)
    for i in range(M):
        for n in range(N):
            assert abs(Fraction(got[i, n]) - want[i][n]) <= abs(want[i][n]) * Fraction(1, 2 ** 45) + Fraction(1, 2 ** 80)


def test_gemm_transpose_pinned_by_permutation():
    K = N = 32
    perm = np.random.default_rng(8).permutation(N)
    codes = np.zeros((N, K), np.uint8)
    codes[np.arange(N), perm] = 0x2          # value 1.0
    scales = np.full((N, K // 16), 0x38, np.uint8)
    qt = O.QTensor(O.pack_codes(codes), scales, 1.0)
    x = np.arange(3 * K, dtype=np.float32).reshape(3, K)
    y = O.gemm_w4a16(x, qt)
    np.testing.assert_array_equal(y, x[:, perm])


def test_full_k16_code_enumeration_single_row():
    # every (code, position) for N=1, K=16 at a random scale: y = sum x_k v_k s
    rng = np.random.default_rng(9)
    x = rng.integers(-8, 9, (1, 16)).astype(np.float32) / 8
    for c in range(16):
        codes = np.full((1, 16), c, np.uint8)
        for sc in (0x01, 0x15, 0x38, 0x7E):
            qt = O.QTensor(O.pack_codes(codes), np.array([[sc]], np.uint8), 0.75)
            want = float(x.astype(np.float64).sum()) * E2M1_TABLE[c & 7] * (-1 if c & 8 else 1) \
                * float(O.e4m3_value(np.array(sc))) * 0.75
            assert O.gemm_w4a16(x, qt)[0, 0] == want


def test_w4a4_uses_decoded_activations():
    rng = np.random.default_rng(10)
    a = rng.standard_t(4, (5, 64)).astype(np.float32)
    w = (rng.standard_normal((7, 64)) * 0.02).astype(np.float32)
    aq, wq = O.quantize(a), O.quantize(w)
    y = O.gemm_w4a4(aq, wq)
    np.testing.assert_allclose(y, O.gemm_w4a16(O.decode(aq), wq), rtol=1e-15, atol=0)
    # and it is a real approximation of the unquantised product
    assert O.rel_fro(y, a.astype(np.float64) @ w.astype(np.float64).T) < 0.2


def test_bf16_round_matches_torch_on_fp32_values():
    rng = np.random.default_rng(11)
    v = rng.standard_normal(100_000).astype(np.float32)
    ties = np.array([1 + 2.0 ** -8, 1 + 3 * 2.0 ** -8, -(1 + 2.0 ** -8), 3 * 2.0 ** -9], np.float32)
    v = np.concatenate([v, ties])
    ref = torch.from_numpy(v).to(torch.bfloat16).to(torch.float64).numpy()
    np.testing.assert_array_equal(O.bf16_round(v.astype(np.float64)), ref)
    assert O.bf16_round(np.array([1 + 2.0 ** -8]))[0] == 1.0


def test_rel_fro():
    assert O.rel_fro(np.array([3.0, 4.0]), np.array([3.0, 4.0])) == 0.0
    assert abs(O.rel_fro(np.array([3.0, 4.5]), np.array([3.0, 4.0])) - 0.1) < 1e-15


# ------------------------------------------------------------- draft head

def _small_head(V=700, K=64, seed=12):
    rng = np.random.default_rng(seed)
    return O.quantize((rng.standard_normal((V, K)) * 0.02).astype(np.float32)), rng


def test_argmax_ties_go_to_lowest_vocab_id():
    logits = np.array([[1.0, 3.0, 3.0, 2.0]])
    rows = np.array([40, 17, 9, 3])
    ids, mx = O.argmax_lowest_id(logits, rows)
    assert ids[0] == 9 and mx[0] == 3.0


def test_masked_head_invariants():
    wq, rng = _small_head()
    V = wq.shape[0]
    idx = rng.permutation(V)[:96]
    h = rng.standard_normal((6, 64))
    full_ids, _, _ = O.gather_gemv_argmax(h, wq, None)
    m_ids, m_max, m_logits = O.gather_gemv_argmax(h, wq, idx)
    for i in range(6):
        assert m_ids[i] in idx
        if full_ids[i] in idx:
            assert m_ids[i] == full_ids[i]
        assert m_max[i] == m_logits[i].max()
    same, _, _ = O.gather_gemv_argmax(h, wq, np.arange(V))
    np.testing.assert_array_equal(same, full_ids)


def test_masked_head_planted_winner():
    wq, rng = _small_head(seed=13)
    idx = rng.permutation(wq.shape[0])[:50]
    h = rng.standard_normal((1, 64))
    target = int(idx[17])
    # plant: row `target` becomes 6*sign(h) in every element at the largest scale
    codes = O.unpack_codes(wq.codes)
    codes[target] = np.where(h[0] >= 0, 0x7, 0xF)
    wq.codes[:] = O.pack_codes(codes)
    wq.scales[target] = 0x7E
    ids, _, _ = O.gather_gemv_argmax(h, wq, idx)
    assert ids[0] == target


def test_greedy_acceptance_hand_cases():
    # target tokens per position, drafts per position (R11): accept up to the first mismatch
    target = np.array([[5, 7, 9, 2], [5, 7, 9, 2], [1, 1, 1, 1], [4, 0, 0, 0]])
    drafts = np.array([[5, 7, 9], [5, 8, 9], [2, 1, 1], [4, 0, 0]])
    np.testing.assert_array_equal(O.accept_greedy(target, drafts), [3, 1, 0, 3])
    # no drafts: every sequence emits just the target token
    np.testing.assert_array_equal(O.accept_greedy(target[:, :1], np.zeros((4, 0), dtype=np.int64)), [0, 0, 0, 0])


def test_verify_accept_drafts_equal_to_the_targets_are_all_accepted():
    wq, rng = _small_head(seed=21)
    B, D = 3, 4
    h = rng.standard_normal((B * (D + 1), 64))
    ids, _, _ = O.gather_gemv_argmax(h, wq, None)
    target = ids.reshape(B, D + 1)
    drafts = target[:, :D].copy()
    # sequence 1: the third draft is wrong; sequence 2: the first one
    drafts[1, 2] = (drafts[1, 2] + 1) % wq.shape[0]
    drafts[2, 0] = (drafts[2, 0] + 5) % wq.shape[0]
    t, n, logits = O.verify_accept(h, wq, drafts)
    np.testing.assert_array_equal(t, target)
    np.testing.assert_array_equal(n, [D, 2, 0])
    assert logits.shape == (B * (D + 1), wq.shape[0])


def test_masked_read_ratio_is_the_pages_7_6x():
    # same bytes per row for every row, so the read shrinks by V / n_idx
    assert round(248320 / 32768, 1) == 7.6


def test_top2_margin():
    m = O.top2_margin(np.array([[0.0, 1.0, 3.0, -4.0]]))
    assert abs(m[0] - 2.0 / np.sqrt(26 / 4)) < 1e-15


# ---------------------------------------------------------------------- MoE

def test_route_matches_sorting():
    rng = np.random.default_rng(14)
    logits = rng.standard_normal((40, 16))
    ids, w = O.moe_route(logits, 4)
    p = torch.softmax(torch.from_numpy(logits), dim=1).numpy()
    for t in range(40):
        order = np.lexsort((np.arange(16), -p[t]))[:4]
        np.testing.assert_array_equal(ids[t], order)
        np.testing.assert_allclose(w[t], p[t, order], rtol=1e-14)
    # a tie in probability goes to the lower expert id
    ids2, _ = O.moe_route(np.array([[0.0, 1.0, 1.0, 0.5]]), 1)
    assert ids2[0, 0] == 1


def _small_moe(T=12, E=4, H=32, I=16, seed=15):
    rng = np.random.default_rng(seed)
    x = torch.from_numpy(rng.standard_normal((T, H)).astype(np.float32)).to(torch.bfloat16).float().numpy()
    w13 = [O.quantize((rng.standard_normal((2 * I, H)) * 0.1).astype(np.float32)) for _ in range(E)]
    w2 = [O.quantize((rng.standard_normal((H, I)) * 0.1).astype(np.float32)) for _ in range(E)]
    return rng, x, w13, w2


def test_moe_top1_reduces_to_dense_layers():
    rng, x, w13, w2 = _small_moe()
    T = x.shape[0]
    ids = np.full((T, 1), 2)
    out = O.moe_forward(x, ids, np.ones((T, 1)), w13, w2)
    gu = O.gemm_w4a16(x, w13[2])
    I = gu.shape[1] // 2
    h = O.bf16_round(gu[:, :I] / (1 + np.exp(-gu[:, :I])) * gu[:, I:])
    np.testing.assert_allclose(out, O.gemm_w4a16(h, w2[2]), rtol=1e-13, atol=1e-15)


def test_moe_is_linear_in_routing_weights_and_permutes_with_tokens():
    rng, x, w13, w2 = _small_moe()
    T = x.shape[0]
    ids, w = O.moe_route(rng.standard_normal((T, 4)), 2)
    out = O.moe_forward(x, ids, w, w13, w2)
    # per-slot decomposition: sum over slots of single-expert layers
    acc = np.zeros_like(out)
    for j in range(2):
        acc += O.moe_forward(x, ids[:, j:j + 1], w[:, j:j + 1], w13, w2)
    np.testing.assert_allclose(out, acc, rtol=1e-13, atol=1e-15)
    perm = rng.permutation(T)
    outp = O.moe_forward(x[perm], ids[perm], w[perm], w13, w2)
    np.testing.assert_allclose(outp, out[perm], rtol=1e-13, atol=1e-15)


# --- R10, W4A4 routed experts ------------------------------------------------

def _moe4_case(seed=21):
    rng, x, w13, w2 = _small_moe(seed=seed)
    T = x.shape[0]
    ids, w = O.moe_route(rng.standard_normal((T, 4)), 2)
    return rng, x, w13, w2, ids, w


def test_moe_w4a4_sees_only_the_quantised_input():
    """Nudging input elements without changing their codes, block scales or
    the tensor scale leaves the layer bit-identical (while the W4A16 layer
    moves), so the input enters only through its quantised form."""
    rng, x, w13, w2, ids, w = _moe4_case()
    q0 = O.quantize(x)
    blocks = np.abs(x).reshape(x.shape[0], -1, 16)
    is_max = (blocks == blocks.max(axis=2, keepdims=True)).reshape(x.shape)
    xn = np.where(is_max, x, x * np.float32(1 + 2.0 ** -14)).astype(np.float32)
    qn = O.quantize(xn)
    # keep only the nudges that leave every code of their block unchanged
    same = (O.unpack_codes(qn.codes) == O.unpack_codes(q0.codes)).reshape(x.shape[0], -1, 16).all(axis=2)
    xn = np.where(np.repeat(same, 16, axis=1), xn, x).astype(np.float32)
    qn = O.quantize(xn)
    assert np.array_equal(qn.codes, q0.codes) and np.array_equal(qn.scales, q0.scales) and qn.s_t == q0.s_t
    assert not np.array_equal(xn, x)
    a = O.moe_forward_w4a4(x, ids, w, w13, w2)
    b = O.moe_forward_w4a4(xn, ids, w, w13, w2)
    assert np.array_equal(a, b)
    assert not np.array_equal(O.moe_forward(x, ids, w, w13, w2), O.moe_forward(xn, ids, w, w13, w2))


def test_moe_w4a4_is_near_the_w4a16_layer_on_the_quantised_input():
    """Against the R7 layer fed the decoded quantised input, only the h
    quantisation differs: a small, non-zero change."""
    rng, x, w13, w2, ids, w = _moe4_case()
    a = O.moe_forward_w4a4(x, ids, w, w13, w2)
    b = O.moe_forward(O.decode(O.quantize(x)), ids, w, w13, w2)
    e = O.rel_fro(a, b)
    assert 0 < e < 0.1


def test_moe_w4a4_h_scale_is_shared_by_all_routed_rows():
    """A token on another expert whose h is the largest of the call changes
    every other token's output (one tensor scale for all h rows); a token
    whose h stays below that maximum changes nothing."""
    rng, x, w13, w2, ids, w = _moe4_case()
    T = x.shape[0]
    ids = np.where(ids == 3, 0, ids)              # the base tokens avoid expert 3
    base = O.moe_forward_w4a4(x, ids, w, w13, w2)
    w13_big = list(w13)
    w13_big[3] = O.quantize((O.decode(w13[3]) * 64).astype(np.float32))
    x_dup = np.concatenate([x, x[:1]])            # same rows: the input's tensor scale is unchanged
    ids_new = np.concatenate([ids, [[3, 3]]])
    w_new = np.concatenate([w, [[0.5, 0.5]]])
    big = O.moe_forward_w4a4(x_dup, ids_new, w_new, w13_big, w2)
    assert not np.array_equal(big[:T], base)
    x_small = np.concatenate([x, x[:1] * np.float32(2.0 ** -6)])
    small = O.moe_forward_w4a4(x_small, ids_new, w_new, w13, w2)
    assert np.array_equal(small[:T], base)


def test_moe_w4a4_permutes_with_tokens_and_scales_with_routing_weights():
    rng, x, w13, w2, ids, w = _moe4_case()
    T = x.shape[0]
    out = O.moe_forward_w4a4(x, ids, w, w13, w2)
    perm = rng.permutation(T)
    np.testing.assert_allclose(O.moe_forward_w4a4(x[perm], ids[perm], w[perm], w13, w2), out[perm],
                               rtol=1e-13, atol=1e-15)
    assert np.array_equal(O.moe_forward_w4a4(x, ids, 2 * w, w13, w2), 2 * out)
