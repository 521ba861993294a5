"""Routed-expert MoE layer: routing kernel and grouped expert GEMMs against
the oracle."""
import numpy as np
import pytest
import torch

import oracle as O
import synth
from tests.gpu_common import DEV, np_f64, nv

pytestmark = pytest.mark.gpu
TOL = 1e-2


# (T, E, k): expert counts held in registers (E <= 128, E <= 256, with lanes
# past E) and the generic kernel (E > 256); token counts off the CTA size
@pytest.mark.parametrize("T,E,k", [(512, 128, 8), (37, 200, 4), (64, 300, 6), (33, 32, 2), (5, 256, 8)])
def test_route_matches_oracle(T, E, k):
    m = nv()
    logits = synth.normal_f32((T, E), 1.0, seed=8 + E)
    ids, w = m.moe_route(logits.to(DEV), k)
    oids, ow = O.moe_route(logits.numpy(), k)
    ids, w = ids.cpu().numpy(), w.cpu().numpy()
    p = torch.softmax(logits.double(), 1).numpy()
    for t in range(T):
        ps = np.sort(p[t])[::-1]
        gaps = np.abs(np.diff(ps[:k + 1]))
        if gaps.min() > 1e-6:            # no near-tie among the top k + 1
            assert list(ids[t]) == list(oids[t])
        assert len(set(ids[t].tolist())) == k and all(0 <= i < E for i in ids[t])
        np.testing.assert_allclose(w[t], p[t, ids[t]], rtol=1e-5)


def moe_case(T, E, H, I, k, seed):
    g = torch.Generator().manual_seed(seed)
    logits = torch.randn(T, E, generator=g)
    x = torch.randn(T, H, generator=g).to(torch.bfloat16)
    w13 = [torch.randn(2 * I, H, generator=g) * 0.02 for _ in range(E)]
    w2 = [torch.randn(H, I, generator=g) * 0.02 for _ in range(E)]
    return logits, x, w13, w2


def oracle_routing(logits, k):
    """The oracle's routing of the router logits, as the grouped GEMM's inputs
    (int32 ids and fp32 weights on the device) and as the oracle's (numpy).
    Both sides of a layer comparison take this one routing; the routing
    kernel is compared with the oracle on its own (test_route_matches_oracle)."""
    oids, ow = O.moe_route(np.asarray(logits, dtype=np.float32), k)
    return (torch.from_numpy(oids.astype(np.int32)).to(DEV), torch.from_numpy(ow.astype(np.float32)).to(DEV),
            oids, ow)


def run_gpu(logits, x, w13, w2, k, ids=None, wts=None):
    m = nv()
    if ids is None:
        ids, wts, _, _ = oracle_routing(logits.numpy(), k)
    q13 = m.quantize_stack([t.to(DEV) for t in w13])
    q2 = m.quantize_stack([t.to(DEV) for t in w2])
    return np_f64(m.grouped_gemm(x.to(DEV), ids, wts, q13, q2)), ids, wts


@pytest.mark.parametrize("T,E,H,I,k", [(16, 4, 128, 128, 2), (100, 8, 256, 128, 3), (37, 16, 128, 256, 8)])
def test_small_layers(T, E, H, I, k):
    logits, x, w13, w2 = moe_case(T, E, H, I, k, seed=T)
    ids, wts, oids, ow = oracle_routing(logits.numpy(), k)
    out, _, _ = run_gpu(logits, x, w13, w2, k, ids, wts)
    ref = O.moe_forward(x.float().numpy(), oids, ow, [O.quantize(t.numpy()) for t in w13],
                        [O.quantize(t.numpy()) for t in w2])
    assert O.rel_fro(out, ref) <= TOL


def test_skewed_routing_all_tokens_to_one_expert():
    T, E, H, I = 70, 4, 128, 128
    logits, x, w13, w2 = moe_case(T, E, H, I, 1, seed=3)
    ids = torch.full((T, 1), 2, dtype=torch.int32, device=DEV)
    wts = torch.ones(T, 1, device=DEV)
    out, _, _ = run_gpu(logits, x, w13, w2, 1, ids, wts)
    ref = O.moe_forward(x.float().numpy(), np.full((T, 1), 2), np.ones((T, 1)),
                        [O.quantize(t.numpy()) for t in w13], [O.quantize(t.numpy()) for t in w2])
    assert O.rel_fro(out, ref) <= TOL


def test_deterministic_across_calls():
    logits, x, w13, w2 = moe_case(64, 8, 128, 128, 4, seed=5)
    a, ids, wts = run_gpu(logits, x, w13, w2, 4)
    b, _, _ = run_gpu(logits, x, w13, w2, 4, ids, wts)
    assert np.array_equal(a, b)


def test_moe_config_t256_sampled_tokens():
    """The 35B-A3B-shaped layer (128 experts, top-8, H=2048, I=768) at T=256:
    64 sampled tokens recomputed by the oracle from its own routing."""
    m = nv()
    T = 256
    logits, x, w13, w2 = synth.moe_inputs(T)
    ids, wts, oids, ow = oracle_routing(logits.numpy(), 8)
    q13 = m.quantize_stack([w13[e].to(DEV) for e in range(128)])
    q2 = m.quantize_stack([w2[e].to(DEV) for e in range(128)])
    out = np_f64(m.grouped_gemm(x.to(DEV), ids, wts, q13, q2))
    toks = np.sort(np.random.default_rng(1).choice(T, 64, replace=False))
    used = sorted(set(oids[toks].ravel().tolist()))
    r13 = {e: O.quantize(w13[e].numpy()) for e in used}
    r2 = {e: O.quantize(w2[e].numpy()) for e in used}
    ref = O.moe_forward(x.float().numpy()[toks], oids[toks], ow[toks],
                        [r13.get(e, r13[used[0]]) for e in range(128)],
                        [r2.get(e, r2[used[0]]) for e in range(128)])
    assert O.rel_fro(out[toks], ref) <= TOL


# With at least 32 routed rows per expert on average (and H, I multiples of
# 256) the expert GEMMs run on the tensor cores: tiles of up to 256 routed
# rows of one expert.
@pytest.mark.parametrize("T,E,H,I,k", [(512, 8, 256, 256, 2), (300, 4, 256, 256, 1), (1024, 4, 256, 512, 2),
                                       (700, 16, 512, 256, 3), (128, 8, 256, 256, 2),
                                       (4096, 4, 256, 256, 2)])
def test_tensor_core_layers(T, E, H, I, k):
    logits, x, w13, w2 = moe_case(T, E, H, I, k, seed=T + 1)
    ids, wts, oids, ow = oracle_routing(logits.numpy(), k)
    out, _, _ = run_gpu(logits, x, w13, w2, k, ids, wts)
    ref = O.moe_forward(x.float().numpy(), oids, ow, [O.quantize(t.numpy()) for t in w13],
                        [O.quantize(t.numpy()) for t in w2])
    assert O.rel_fro(out, ref) <= TOL


def test_tensor_core_skewed_routing_ragged_tiles():
    """600 rows on one expert: three tiles of 200 rows (the plan splits an expert evenly into
    tiles of at most 256, rounded up to 32 rows); the other experts get none."""
    T, E, H, I = 600, 4, 256, 256
    logits, x, w13, w2 = moe_case(T, E, H, I, 1, seed=11)
    ids = torch.full((T, 1), 1, dtype=torch.int32, device=DEV)
    wts = torch.full((T, 1), 0.5, device=DEV)
    out, _, _ = run_gpu(logits, x, w13, w2, 1, ids, wts)
    ref = O.moe_forward(x.float().numpy(), np.full((T, 1), 1), np.full((T, 1), 0.5),
                        [O.quantize(t.numpy()) for t in w13], [O.quantize(t.numpy()) for t in w2])
    assert O.rel_fro(out, ref) <= TOL


def test_tensor_core_deterministic_and_scaled_tokens():
    """Repeatable bit for bit; tokens whose magnitudes span 2^-20..2^20 (the
    per-row power-of-two shift of the f16 copies)."""
    T, E, H, I, k = 512, 4, 256, 256, 2
    logits, x, w13, w2 = moe_case(T, E, H, I, k, seed=13)
    scale = torch.pow(2.0, torch.linspace(-20, 20, T)).unsqueeze(1)
    x = (x.float() * scale).to(torch.bfloat16)
    ids, wts, oids, ow = oracle_routing(logits.numpy(), k)
    a, _, _ = run_gpu(logits, x, w13, w2, k, ids, wts)
    b, _, _ = run_gpu(logits, x, w13, w2, k, ids, wts)
    assert np.array_equal(a, b)
    ref = O.moe_forward(x.float().numpy(), oids, ow, [O.quantize(t.numpy()) for t in w13],
                        [O.quantize(t.numpy()) for t in w2])
    # per-token relative error: the rows span 40 binades
    for t in range(0, T, 37):
        assert O.rel_fro(a[t], ref[t]) <= TOL


def test_moe_config_t4096_sampled_tokens():
    """The 35B-A3B-shaped layer at T=4096 (256 routed rows per expert on
    average: the tensor-core path), 32 sampled tokens against the oracle."""
    m = nv()
    T = 4096
    logits, x, w13, w2 = synth.moe_inputs(T)
    ids, wts, oids, ow = oracle_routing(logits.numpy(), 8)
    q13 = m.quantize_stack([w13[e].to(DEV) for e in range(128)])
    q2 = m.quantize_stack([w2[e].to(DEV) for e in range(128)])
    out = np_f64(m.grouped_gemm(x.to(DEV), ids, wts, q13, q2))
    toks = np.sort(np.random.default_rng(2).choice(T, 32, replace=False))
    used = sorted(set(oids[toks].ravel().tolist()))
    r13 = {e: O.quantize(w13[e].numpy()) for e in used}
    r2 = {e: O.quantize(w2[e].numpy()) for e in used}
    ref = O.moe_forward(x.float().numpy()[toks], oids[toks], ow[toks],
                        [r13.get(e, r13[used[0]]) for e in range(128)],
                        [r2.get(e, r2[used[0]]) for e in range(128)])
    assert O.rel_fro(out[toks], ref) <= TOL


@pytest.mark.parametrize("T,E,H,I", [(40, 8, 128, 128), (512, 4, 256, 256), (4096, 4, 256, 256)])
def test_out_of_range_expert_ids_are_dropped_and_reported(T, E, H, I):
    """Slots whose expert id is -2, -1 or E contribute nothing, and the call
    reports NVFP4_ERR_INVALID_ARG in the device status word; the result equals
    the layer with those slots' weights set to zero. (512, 4, 256, 256) runs the
    tensor-core path; (4096, 4, 256, 256), 8192 routed slots, also the
    routing plan over several CTAs."""
    m = nv()
    k = 2
    logits, x, w13, w2 = moe_case(T, E, H, I, k, seed=T + 7)
    ids, wts, _, _ = oracle_routing(logits.numpy(), k)
    bad = ids.clone()
    bad[0, 0], bad[3, 1], bad[T - 1, 0] = -2, -1, E
    dropped = wts.clone()
    dropped[0, 0], dropped[3, 1], dropped[T - 1, 0] = 0.0, 0.0, 0.0
    m.read_device_status()   # clear
    out, _, _ = run_gpu(logits, x, w13, w2, k, bad, wts)
    assert m.read_device_status() == m.ERR_INVALID_ARG
    assert np.all(np.isfinite(out))
    ref_ids = bad.cpu().numpy()
    ref = O.moe_forward(x.float().numpy(), ref_ids, dropped.cpu().numpy().astype(np.float64),
                        [O.quantize(t.numpy()) for t in w13], [O.quantize(t.numpy()) for t in w2])
    assert O.rel_fro(out, ref) <= TOL
    # the same as routing those slots to a real expert with weight zero
    ok_ids = ids.clone()
    clean, _, _ = run_gpu(logits, x, w13, w2, k, ok_ids, dropped)
    assert m.read_device_status() == m.OK
    assert O.rel_fro(out, clean) <= TOL


# ---------------------------------------------------------------------------
# The same layer with 4-bit activations (W4A4, reading R10): experts' scales
# prepacked into the MMA layout, against oracle.moe_forward_w4a4.

def run_gpu_w4a4(x, w13, w2, ids, wts):
    m = nv()
    q13 = m.prepack_scales(m.quantize_stack([t.to(DEV) for t in w13]))
    q2 = m.prepack_scales(m.quantize_stack([t.to(DEV) for t in w2]))
    return np_f64(m.grouped_gemm_w4a4(x.to(DEV), ids, wts, q13, q2))


def ref_w4a4(x, w13, w2, ids, wts):
    return O.moe_forward_w4a4(x.float().numpy(), ids.cpu().numpy(), wts.cpu().numpy().astype(np.float64),
                              [O.quantize(t.numpy()) for t in w13], [O.quantize(t.numpy()) for t in w2])


# the last three: 256+ routed rows per expert on average, so the expert GEMMs
# run on CTA pairs over 256-row tiles (ragged tiles included)
@pytest.mark.parametrize("T,E,H,I,k", [(64, 4, 256, 128, 2), (300, 8, 512, 256, 3), (37, 16, 256, 384, 8),
                                       (1, 4, 256, 128, 1), (700, 4, 256, 256, 2), (1024, 4, 256, 256, 2),
                                       (700, 2, 256, 384, 1), (2048, 8, 512, 256, 2)])
def test_w4a4_layers(T, E, H, I, k):
    """Ragged tiles (several 128-row tiles per expert, ragged tails), one
    token, top-8, I not a multiple of 256 (three-atom last K stage)."""
    logits, x, w13, w2 = moe_case(T, E, H, I, k, seed=T + 31)
    ids, wts, _, _ = oracle_routing(logits.numpy(), k)
    out = run_gpu_w4a4(x, w13, w2, ids, wts)
    assert O.rel_fro(out, ref_w4a4(x, w13, w2, ids, wts)) <= TOL


@pytest.mark.parametrize("E", [4, 2])
def test_w4a4_skewed_routing_and_determinism(E):
    """600 rows on one expert, the others empty; two calls give identical bits.
    E = 4: one-CTA kernels, five 120-row tiles; E = 2 (300 rows per expert on
    average): CTA pairs, three 200-row tiles, each with a ragged odd half."""
    T, H, I = 600, 256, 256
    logits, x, w13, w2 = moe_case(T, E, H, I, 1, seed=41)
    ids = torch.full((T, 1), E - 1, dtype=torch.int32, device=DEV)
    wts = torch.full((T, 1), 0.75, device=DEV)
    a = run_gpu_w4a4(x, w13, w2, ids, wts)
    b = run_gpu_w4a4(x, w13, w2, ids, wts)
    assert np.array_equal(a, b)
    assert O.rel_fro(a, ref_w4a4(x, w13, w2, ids, wts)) <= TOL


def test_w4a4_out_of_range_expert_ids_are_dropped_and_reported():
    m = nv()
    T, E, H, I, k = 96, 4, 256, 128, 2
    logits, x, w13, w2 = moe_case(T, E, H, I, k, seed=43)
    ids, wts, _, _ = oracle_routing(logits.numpy(), k)
    bad = ids.clone()
    bad[0, 1], bad[5, 0], bad[T - 1, 1] = -2, E, -1
    m.read_device_status()
    out = run_gpu_w4a4(x, w13, w2, bad, wts)
    assert m.read_device_status() == m.ERR_INVALID_ARG
    assert np.all(np.isfinite(out))
    assert O.rel_fro(out, ref_w4a4(x, w13, w2, bad, wts)) <= TOL


def test_w4a4_moe_config_t4096_sampled_tokens():
    """The 35B-A3B-shaped layer (128 experts, top-8, H=2048, I=768) at
    T=4096 with 4-bit activations: the oracle runs the whole layer (the h
    rows' tensor scale depends on every routed row) with the experts
    quantised in spawned workers; 64 sampled tokens compared."""
    from tests.moe_oracle import quantize_experts
    m = nv()
    T = 4096
    logits, x, w13, w2 = synth.moe_inputs(T)
    ids, wts, oids, ow = oracle_routing(logits.numpy(), 8)
    q13 = m.prepack_scales(m.quantize_stack([w13[e].to(DEV) for e in range(128)]))
    q2 = m.prepack_scales(m.quantize_stack([w2[e].to(DEV) for e in range(128)]))
    out = np_f64(m.grouped_gemm_w4a4(x.to(DEV), ids, wts, q13, q2))
    r13 = quantize_experts(w13.numpy())
    r2 = quantize_experts(w2.numpy())
    ref = O.moe_forward_w4a4(x.float().numpy(), oids, ow, r13, r2)
    toks = np.sort(np.random.default_rng(3).choice(T, 64, replace=False))
    assert O.rel_fro(out[toks], ref[toks]) <= TOL
