"""Pins of the CPU oracle against facts that do not come from the oracle itself.

Every check here compares the oracle with something independent: values printed
on the pages (tests/golden), library routines (ml_dtypes, torch, scipy),
exact rational arithmetic, brute force on tiny inputs, or invariants of the
mathematics.  None of these tests needs a GPU.
"""

from fractions import Fraction

import numpy as np
import pytest
import torch

import synth
from oracle import formats, moe, requant, route
from tests.exact_fp32 import f32, round_fp32

# ----------------------------------------------------------------------------- formats


def test_e2m1_all_16_codes_match_ml_dtypes():
    ml_dtypes = pytest.importorskip("ml_dtypes")
    codes = np.arange(16, dtype=np.uint8)
    lib = codes.view(ml_dtypes.float4_e2m1fn).astype(np.float64)
    ours = formats.e2m1_decode(codes)
    assert np.array_equal(np.signbit(lib), np.signbit(ours))
    assert np.array_equal(lib, ours)


def test_e2m1_closed_form_facts():
    v = formats.e2m1_decode(np.arange(16))
    # largest magnitude 6 (E2M1 emax = 2, mantissa 1.5), smallest subnormal 0.5,
    # code 8 is negative zero, the upper 8 codes mirror the lower 8.
    assert v.max() == 6.0 and v.min() == -6.0
    assert v[1] == 0.5 and v[0] == 0.0
    assert v[8] == 0.0 and np.signbit(v[8])
    assert np.array_equal(v[8:], -v[:8])
    assert np.all(np.diff(v[:8]) > 0)


def test_e8m0_all_256_codes_match_torch():
    b = torch.arange(256, dtype=torch.int32).to(torch.uint8)
    lib = b.view(torch.float8_e8m0fnu).to(torch.float64).numpy()
    ours = formats.e8m0_decode(b.numpy())
    assert np.isnan(ours[255]) and np.isnan(lib[255])
    assert np.array_equal(lib[:255], ours[:255])
    assert ours[127] == 1.0 and ours[0] == 2.0 ** -127 and ours[254] == 2.0 ** 127


def test_nibble_order_and_pack_roundtrip():
    # Byte 0x21 holds element 0 = code 1 (low nibble) and element 1 = code 2.
    assert list(formats.unpack_nibbles(np.array([0x21], np.uint8))) == [1, 2]
    g = np.random.default_rng(0)
    codes = g.integers(0, 16, size=(3, 5, 64), dtype=np.uint8)
    assert np.array_equal(formats.unpack_nibbles(formats.pack_nibbles(codes)), codes)


def test_dequant_elementwise_against_libraries():
    ml_dtypes = pytest.importorskip("ml_dtypes")
    g = np.random.default_rng(1)
    packed = g.integers(0, 256, size=(2, 3, 32), dtype=np.uint8)  # K = 64
    scales = g.integers(100, 150, size=(2, 3, 2), dtype=np.uint8)
    ours = formats.dequant_mxfp4(packed, scales)
    lo = (packed & 0xF).view(ml_dtypes.float4_e2m1fn).astype(np.float64)
    hi = (packed >> 4).view(ml_dtypes.float4_e2m1fn).astype(np.float64)
    sc = torch.from_numpy(scales).view(torch.float8_e8m0fnu).to(torch.float64).numpy()
    for e in range(2):
        for n in range(3):
            for k in range(64):
                code_val = lo[e, n, k // 2] if k % 2 == 0 else hi[e, n, k // 2]
                assert ours[e, n, k] == code_val * sc[e, n, k // 32]


def test_byte_layouts_match_printed_shapes(golden):
    f = golden("k3_layouts.txt")
    H, I = f["model_dim"], f["intermediate_dim"]
    # create_weights: w13 [E, 2*I_partition, H/2]; printed per-rank TP8 shape (896, 768, 1792)
    assert [f["global_experts"], 2 * I // f["tp"], H // 2] == f["w13_tp8_shape"]
    # round-up to 256 per partition: 384 -> 512 rows per half
    assert [f["global_experts"], 2 * 512, H // 2] == f["w13_tp8_roundup_shape"]
    assert f["global_experts"] // f["tp"] == f["local_experts"]
    assert formats.MX_BLOCK == f["mxfp4_block"]
    # a packed byte holds two elements; float32 decode is 8 bytes per packed byte
    packed = np.zeros((1, 4, H // 2), np.uint8)
    sc = np.full((1, 4, H // 32), 127, np.uint8)
    deq = formats.dequant_mxfp4(packed, sc).astype(np.float32)
    assert deq.nbytes == f["unpack_growth"] * packed.nbytes
    assert deq.shape == (1, 4, H)


def test_bf16_helpers_against_torch():
    g = np.random.default_rng(2)
    a = (g.standard_normal(4096) * np.exp(g.uniform(-30, 30, 4096))).astype(np.float32)
    ours = formats.f32_to_bf16_rne(a)
    lib = torch.from_numpy(a).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    assert np.array_equal(ours, lib)
    back = formats.bf16_to_f64(lib)
    assert np.array_equal(back, torch.from_numpy(lib.view(np.int16)).view(torch.bfloat16).double().numpy())


# ----------------------------------------------------------------------------- MXFP4 quantiser (input synthesis)


def test_quantiser_roundtrip_on_grid_blocks():
    # Blocks whose largest magnitude is code 6 or 7 (value 4 or 6) are fixed
    # points of quantise(dequantise(.)): the floor rule maps their amax into [4, 8).
    g = np.random.default_rng(3)
    codes = g.integers(0, 16, size=(64, 32), dtype=np.uint8)
    codes[:, 0] = np.where(g.integers(0, 2, 64) == 0, 6, 7) | (g.integers(0, 2, 64).astype(np.uint8) << 3)
    codes[:, 1:] = np.where((codes[:, 1:] & 7) > 5, codes[:, 1:] & 8, codes[:, 1:])  # keep others < amax
    packed = formats.pack_nibbles(codes)
    sc = g.integers(60, 200, size=(64, 1), dtype=np.uint8)
    w = formats.dequant_mxfp4(packed, sc)
    p2, s2 = formats.quantize_mxfp4(w)
    assert np.array_equal(s2, sc)
    # -0 and +0 both decode to 0; compare decoded values
    assert np.array_equal(formats.dequant_mxfp4(p2, s2), w)


def test_quantiser_error_bound():
    g = np.random.default_rng(4)
    w = g.standard_normal((16, 256)) * 0.02
    p, s = formats.quantize_mxfp4(w)
    d = formats.dequant_mxfp4(p, s)
    X = formats.e8m0_decode(s).repeat(32, axis=1)
    r = np.abs(w) / X
    # half of the local grid spacing: 0.25 below 2, 0.5 in [2, 4), 1 in [4, 6]
    step = np.where(r < 2, 0.5, np.where(r < 4, 1.0, 2.0))
    inside = r <= 6
    assert np.all(np.abs(d - w)[inside] <= (step / 2 * X)[inside] + 1e-18)
    assert np.all(np.abs(d[~inside]) == 6 * X[~inside])


# ----------------------------------------------------------------------------- routing


def _route_bruteforce(ids, E):
    P = ids.size
    flat = ids.reshape(-1)
    counts = [0] * E
    lists = [[] for _ in range(E)]
    for p in range(P):
        e = int(flat[p])
        if 0 <= e < E:
            counts[e] += 1
            lists[e].append(p)
    sp = [p for e in range(E) for p in lists[e]]
    pos = [-1] * P
    for i, p in enumerate(sp):
        pos[p] = i
    sp += [-1] * (P - len(sp))
    offs = [0]
    for c in counts:
        offs.append(offs[-1] + c)
    return counts, offs, sp, pos


@pytest.mark.parametrize("T,topk,E", [(1, 15, 112), (7, 15, 112), (33, 4, 8), (5, 3, 2)])
def test_route_matches_bruteforce_with_invalid_and_duplicate_ids(T, topk, E):
    g = np.random.default_rng(T * 100 + topk)
    ids = g.integers(-2, E + 2, size=(T, topk)).astype(np.int32)
    c, o, sp, pos = route.route(ids, E)
    bc, bo, bsp, bpos = _route_bruteforce(ids, E)
    assert list(c) == bc and list(o) == bo and list(sp) == bsp and list(pos) == bpos


@pytest.mark.parametrize("G,E", [(16, 8), (9, 3)])
def test_route_with_expert_map_matches_bruteforce(G, E):
    # global ids (some out of range) through a map that sends some experts to
    # other GPUs (-1): the brute force maps each id by hand, then groups
    g = np.random.default_rng(G * 10 + E)
    ids = g.integers(-2, G + 2, size=(11, 4)).astype(np.int32)
    emap = np.full(G, -1, np.int32)
    owned = g.choice(G, E, replace=False)
    emap[owned] = g.permutation(E)
    local = [[int(emap[i]) if 0 <= i < G else -1 for i in row] for row in ids]
    c, o, sp, pos = route.route(ids, E, expert_map=emap)
    bc, bo, bsp, bpos = _route_bruteforce(np.array(local, np.int32), E)
    assert list(c) == bc and list(o) == bo and list(sp) == bsp and list(pos) == bpos


def test_router_topk_against_scipy_softmax_and_bruteforce():
    # scipy's softmax, then a brute-force selection: k passes, each taking the
    # largest remaining probability (the first such id on ties)
    from scipy.special import softmax

    g = np.random.default_rng(41)
    logits = g.standard_normal((6, 40)).astype(np.float32)
    logits[2, [3, 9, 17]] = 2.5  # a three-way tie at the top
    for renorm in (True, False):
        ids, w = route.router_topk(logits, 5, renormalize=renorm)
        for t in range(logits.shape[0]):
            p = softmax(logits[t].astype(np.float64))
            left = list(range(logits.shape[1]))
            want = []
            for _ in range(5):
                best = max(left, key=lambda i: (p[i], -i))
                want.append(best)
                left.remove(best)
            assert list(ids[t]) == want
            pw = p[want] / (p[want].sum() if renorm else 1.0)
            assert np.allclose(w[t], pw.astype(np.float32), rtol=1e-6, atol=0)
    assert list(route.router_topk(logits, 5)[0][2][:3]) == [3, 9, 17]


def test_router_topk_invariants():
    g = np.random.default_rng(42)
    logits = g.standard_normal((5, 16))
    ids, w = route.router_topk(logits, 4)
    assert np.allclose(w.sum(axis=1), 1.0, atol=1e-6)
    assert np.all(np.diff(w, axis=1) <= 0)  # decreasing weights
    ids2, w2 = route.router_topk(logits + 7.25, 4)  # softmax is shift invariant
    assert np.array_equal(ids, ids2) and np.allclose(w, w2, rtol=1e-6)
    ids_all, _ = route.router_topk(logits, 16)  # k = all experts: a permutation
    assert all(sorted(r) == list(range(16)) for r in ids_all)
    one_hot = np.full((2, 8), -30.0)
    one_hot[0, 5] = one_hot[1, 2] = 30.0
    ids1, w1 = route.router_topk(one_hot, 1, renormalize=False)
    assert list(ids1[:, 0]) == [5, 2] and np.allclose(w1, 1.0)


def test_route_empty():
    c, o, sp, pos = route.route(np.zeros((0, 4), np.int32), 8)
    assert c.sum() == 0 and o[-1] == 0 and sp.size == 0 and pos.size == 0


# ----------------------------------------------------------------------------- MoE forward


def test_silu_against_scipy():
    special = pytest.importorskip("scipy.special")
    z = np.linspace(-40, 40, 1001)
    assert np.allclose(moe.silu(z), z * special.expit(z), rtol=1e-15, atol=1e-300)


def _tiny_problem(seed, E=8, H=64, I=64, T=5, topk=2):
    g = synth.rng(seed)
    x = synth.activations_bf16(g, T, H)
    ids, w = synth.router_topk(g, T, E, topk)
    w13, s13 = formats.quantize_mxfp4(synth.gaussian(g, (E, 2 * I, H), 0.02))
    w2, s2 = formats.quantize_mxfp4(synth.gaussian(g, (E, H, I), 0.02))
    return x, ids, w, w13, s13, w2, s2


def _dense_torch(x, ids, w, w13, s13, w2, s2):
    """Every expert on every token with torch float64 ops, then the top-k mask."""
    X = torch.from_numpy(x.view(np.int16)).view(torch.bfloat16).double()
    W13 = torch.from_numpy(formats.dequant_mxfp4(w13, s13))
    W2 = torch.from_numpy(formats.dequant_mxfp4(w2, s2))
    I = W13.shape[1] // 2
    h = torch.einsum("eih,th->eti", W13, X)
    a = torch.nn.functional.silu(h[..., :I]) * h[..., I:]
    Y = torch.einsum("ehi,eti->eth", W2, a)  # [E, T, H]
    E = W13.shape[0]
    mask = torch.zeros(E, X.shape[0], dtype=torch.float64)
    for t in range(ids.shape[0]):
        for k in range(ids.shape[1]):
            if 0 <= ids[t, k] < E:
                mask[ids[t, k], t] += float(w[t, k])
    return torch.einsum("et,eth->th", mask, Y).numpy()


@pytest.mark.parametrize("seed", [0, 1, 2])
def test_moe_matches_dense_bruteforce(seed):
    x, ids, w, w13, s13, w2, s2 = _tiny_problem(seed)
    ours = moe.moe_forward(x, ids, w, w13, s13, w2, s2)
    ref = _dense_torch(x, ids, w, w13, s13, w2, s2)
    assert np.allclose(ours, ref, rtol=1e-12, atol=1e-14)


def test_moe_dense_bruteforce_with_invalid_and_duplicate_ids():
    x, ids, w, w13, s13, w2, s2 = _tiny_problem(7, T=6, topk=3)
    ids[0, 1] = -1
    ids[1, 2] = 99
    ids[2, :] = 3  # the same expert three times
    ours = moe.moe_forward(x, ids, w, w13, s13, w2, s2)
    ref = _dense_torch(x, ids, w, w13, s13, w2, s2)
    assert np.allclose(ours, ref, rtol=1e-12, atol=1e-14)


def test_moe_single_expert_is_textbook_swiglu_mlp():
    x, ids, w, w13, s13, w2, s2 = _tiny_problem(5, E=1, T=3, topk=1)
    ids[:] = 0
    w[:] = 1.0
    ours = moe.moe_forward(x, ids, w, w13, s13, w2, s2)
    X = torch.from_numpy(x.view(np.int16)).view(torch.bfloat16).double()
    W13 = torch.from_numpy(formats.dequant_mxfp4(w13, s13))[0]
    W2 = torch.from_numpy(formats.dequant_mxfp4(w2, s2))[0]
    I = W13.shape[0] // 2
    gate = torch.nn.functional.linear(X, W13[:I])
    up = torch.nn.functional.linear(X, W13[I:])
    ref = torch.nn.functional.linear(torch.nn.functional.silu(gate) * up, W2)
    assert np.allclose(ours, ref.numpy(), rtol=1e-12, atol=1e-14)


def test_moe_invariants():
    x, ids, w, w13, s13, w2, s2 = _tiny_problem(9)
    base = moe.moe_forward(x, ids, w, w13, s13, w2, s2)
    # linear in the router weights
    assert np.allclose(moe.moe_forward(x, ids, w * 2, w13, s13, w2, s2), 2 * base, rtol=1e-12)
    assert np.all(moe.moe_forward(x, ids, w * 0, w13, s13, w2, s2) == 0)
    # relabelling the experts (and their weights) changes nothing
    perm = np.random.default_rng(0).permutation(w13.shape[0])
    inv = np.argsort(perm)
    out = moe.moe_forward(x, inv[ids].astype(np.int32), w, w13[perm], s13[perm], w2[perm], s2[perm])
    assert np.allclose(out, base, rtol=1e-12, atol=1e-15)
    # zero input gives zero output (SiLU(0) = 0)
    assert np.all(moe.moe_forward(np.zeros_like(x), ids, w, w13, s13, w2, s2) == 0)


def _bias_bits(g, shape, std=0.5):
    return synth.bf16_bits_from_f32(synth.gaussian(g, shape, std))


def _dense_torch_variants(x, ids, w, w13, s13, w2, s2, b13, b2, on_input):
    """Every expert on every token through torch's linear-with-bias, then the
    top-k selection (router weight on the input or on the output)."""
    X = torch.from_numpy(x.view(np.int16)).view(torch.bfloat16).double()
    W13 = torch.from_numpy(formats.dequant_mxfp4(w13, s13))
    W2 = torch.from_numpy(formats.dequant_mxfp4(w2, s2))
    B13 = torch.from_numpy(b13.view(np.int16)).view(torch.bfloat16).double()
    B2 = torch.from_numpy(b2.view(np.int16)).view(torch.bfloat16).double()
    E, I = W13.shape[0], W13.shape[1] // 2
    out = torch.zeros(X.shape, dtype=torch.float64)
    for t in range(ids.shape[0]):
        for k in range(ids.shape[1]):
            e = int(ids[t, k])
            if not 0 <= e < E:
                continue
            xt = X[t] * float(w[t, k]) if on_input else X[t]
            h = torch.nn.functional.linear(xt, W13[e], B13[e])
            a = torch.nn.functional.silu(h[:I]) * h[I:]
            y = torch.nn.functional.linear(a, W2[e], B2[e])
            out[t] += y if on_input else float(w[t, k]) * y
    return out.numpy()


@pytest.mark.parametrize("on_input", [False, True])
def test_moe_bias_and_router_weight_on_input_match_torch_linear(on_input):
    x, ids, w, w13, s13, w2, s2 = _tiny_problem(21, T=6, topk=3)
    ids[1, 2] = -1
    g = synth.rng(22)
    E, I2, H = w13.shape[0], w13.shape[1], w2.shape[1]
    b13, b2 = _bias_bits(g, (E, I2)), _bias_bits(g, (E, H))
    ours = moe.moe_forward(x, ids, w, w13, s13, w2, s2, b13=b13, b2=b2, router_weight_on_input=on_input)
    ref = _dense_torch_variants(x, ids, w, w13, s13, w2, s2, b13, b2, on_input)
    assert np.allclose(ours, ref, rtol=1e-12, atol=1e-14)


def test_moe_bias_closed_form_with_zero_weights():
    # all-zero E2M1 codes: h = b13, y = b2, so out[t] = sum_k w[t,k] * b2[e]
    # (router weight on the output) or sum_k b2[e] (router weight on the input)
    x, ids, w, w13, s13, w2, s2 = _tiny_problem(23, T=5, topk=2)
    ids[3, 1] = 8  # invalid
    g = synth.rng(24)
    E, I2, H = w13.shape[0], w13.shape[1], w2.shape[1]
    b13, b2 = _bias_bits(g, (E, I2)), _bias_bits(g, (E, H))
    z13, z2 = np.zeros_like(w13), np.zeros_like(w2)
    B2 = formats.bf16_to_f64(b2)
    want_w = np.zeros((ids.shape[0], H))
    want_1 = np.zeros((ids.shape[0], H))
    for t in range(ids.shape[0]):
        for k in range(ids.shape[1]):
            if 0 <= ids[t, k] < E:
                want_w[t] += float(w[t, k]) * B2[ids[t, k]]
                want_1[t] += B2[ids[t, k]]
    got_w = moe.moe_forward(x, ids, w, z13, s13, z2, s2, b13=b13, b2=b2)
    got_1 = moe.moe_forward(x, ids, w, z13, s13, z2, s2, b13=b13, b2=b2, router_weight_on_input=True)
    assert np.array_equal(got_w, want_w)
    assert np.array_equal(got_1, want_1)
    # without biases the same weights give zero
    assert np.all(moe.moe_forward(x, ids, w, z13, s13, z2, s2) == 0)


def test_moe_expert_map_partition_sums_to_the_whole_layer():
    # expert parallelism: 8 global experts split over two GPUs by parity (local
    # id = global // 2); each GPU maps the ids it does not hold to -1, and the
    # two partial outputs add up to the layer computed with every expert local
    x, ids, w, w13, s13, w2, s2 = _tiny_problem(31, T=7, topk=3)
    G = w13.shape[0]
    whole = moe.moe_forward(x, ids, w, w13, s13, w2, s2)
    parts = []
    for r in range(2):
        held = np.arange(r, G, 2)
        emap = np.full(G, -1, np.int32)
        emap[held] = np.arange(held.size)
        parts.append(moe.moe_forward(x, ids, w, w13[held], s13[held], w2[held], s2[held], expert_map=emap))
    assert np.allclose(parts[0] + parts[1], whole, rtol=1e-12, atol=1e-14)
    # a map that holds nothing gives zero; the identity map changes nothing
    none = np.full(G, -1, np.int32)
    assert np.all(moe.moe_forward(x, ids, w, w13, s13, w2, s2, expert_map=none) == 0)
    ident = np.arange(G, dtype=np.int32)
    assert np.array_equal(moe.moe_forward(x, ids, w, w13, s13, w2, s2, expert_map=ident), whole)


def test_moe_sampled_matches_full():
    x, ids, w, w13, s13, w2, s2 = _tiny_problem(11, T=9, topk=3)
    full = moe.moe_forward(x, ids, w, w13, s13, w2, s2)
    toks, cols = np.array([0, 4, 8]), np.array([0, 5, 17, 63])
    samp = moe.moe_forward_sampled(x, ids, w, w13, s13, w2, s2, toks, cols)
    assert np.allclose(samp, full[np.ix_(toks, cols)], rtol=1e-12, atol=1e-15)


def test_int4_dequant_bruteforce():
    g = np.random.default_rng(12)
    q = g.integers(0, 256, size=(2, 3, 16), dtype=np.uint8)  # K = 32
    s = g.standard_normal((2, 3, 1)).astype(np.float32)
    d = moe.dequant_int4(q, s)
    for e in range(2):
        for n in range(3):
            for k in range(32):
                nib = (int(q[e, n, k // 2]) >> (4 * (k % 2))) & 0xF
                val = nib - 16 if nib >= 8 else nib
                assert d[e, n, k] == val * float(s[e, n, 0])


# ----------------------------------------------------------------------------- requantiser


def _requant_exact(vals_f64, K, bf16_scale=False):
    """Exact-rational restatement of the int4 rule on decoded values (one row);
    with ``bf16_scale`` the scale is rounded on to bfloat16 (8 significant bits)
    before the elements are divided by it."""
    q = []
    scales = []
    for g0 in range(0, K, 32):
        blk = [Fraction(float(v)) for v in vals_f64[g0:g0 + 32]]
        amax = max(abs(b) for b in blk)
        sc = round_fp32(amax / 7)
        if bf16_scale:
            sc = round_fp32(sc, mant_bits=7)
        scales.append(sc)
        for b in blk:
            if sc == 0:
                q.append(0)
            else:
                q.append(max(-8, min(7, round(round_fp32(b / sc)))))
    return q, scales


@pytest.mark.parametrize("s_lo,s_hi", [(0, 6), (100, 130), (245, 252)])
def test_requant_matches_exact_rational_ieee(s_lo, s_hi):
    g = np.random.default_rng(s_lo)
    E, N, K = 2, 3, 64
    w = g.integers(0, 256, size=(E, N, K // 2), dtype=np.uint8)
    w[0, 0, :16] = 0  # an all-zero group
    sc = g.integers(s_lo, s_hi + 1, size=(E, N, K // 32), dtype=np.uint8)
    oq, os_ = requant.requant_mxfp4_to_int4g32(w, sc)
    vals = formats.dequant_mxfp4(w, sc)
    for e in range(E):
        for n in range(N):
            q_ref, s_ref = _requant_exact(vals[e, n], K)
            codes = formats.unpack_nibbles(oq[e, n]).astype(np.int64)
            q_got = np.where(codes >= 8, codes - 16, codes)
            assert list(q_got) == q_ref
            assert [f32(v) for v in os_[e, n]] == s_ref


@pytest.mark.parametrize("s_lo,s_hi", [(0, 6), (100, 130), (245, 252)])
def test_requant_bf16_scales_match_exact_rational_ieee(s_lo, s_hi):
    g = np.random.default_rng(s_lo + 7)
    E, N, K = 2, 3, 96
    w = g.integers(0, 256, size=(E, N, K // 2), dtype=np.uint8)
    w[1, 2, 16:32] = 0  # an all-zero group
    sc = g.integers(s_lo, s_hi + 1, size=(E, N, K // 32), dtype=np.uint8)
    oq, os_ = requant.requant_mxfp4_to_int4g32(w, sc, scale_dtype="bf16")
    assert os_.dtype == np.uint16
    vals = formats.dequant_mxfp4(w, sc)
    for e in range(E):
        for n in range(N):
            q_ref, s_ref = _requant_exact(vals[e, n], K, bf16_scale=True)
            codes = formats.unpack_nibbles(oq[e, n]).astype(np.int64)
            assert list(np.where(codes >= 8, codes - 16, codes)) == q_ref
            assert [Fraction(float(v)) for v in formats.bf16_to_f64(os_[e, n])] == s_ref


def test_requant_bf16_scales_differ_from_f32_and_stay_in_range():
    g = np.random.default_rng(33)
    w = g.integers(0, 256, size=(4, 16, 128), dtype=np.uint8)
    sc = g.integers(100, 140, size=(4, 16, 8), dtype=np.uint8)
    q32, s32 = requant.requant_mxfp4_to_int4g32(w, sc)
    qb, sb = requant.requant_mxfp4_to_int4g32(w, sc, scale_dtype="bf16")
    sbf = formats.bf16_to_f64(sb)
    # the stored scale is the float32 one rounded to bf16 (8 significant bits:
    # relative change <= 2^-8)
    assert np.array_equal(sbf, formats.bf16_to_f64(formats.f32_to_bf16_rne(s32)))
    assert np.all(np.abs(sbf - s32) <= 2.0 ** -8 * s32)
    assert not np.array_equal(sbf, s32.astype(np.float64))
    codes = formats.unpack_nibbles(qb).astype(np.int64)
    q = np.where(codes >= 8, codes - 16, codes)
    assert q.min() >= -7 and q.max() <= 7
    # dequantisation through the MoE oracle's bf16-scale kind uses the stored scale
    deq = moe._deq("int4g32_bf16", qb[0], sb[0])
    assert np.array_equal(deq, moe.dequant_int4(qb[0], sbf[0].astype(np.float32)))


def test_requant_all_code_pairs_scale_invariant():
    # Within the normal float32 range q depends only on (element code, block max code).
    table = {}
    for s in (5, 8, 60, 127, 200, 252):
        for cmax in range(1, 8):
            for c in range(16):
                if (c & 7) > cmax:
                    continue
                codes = np.zeros(32, np.uint8)
                codes[0] = cmax
                codes[1] = c
                w = formats.pack_nibbles(codes)[None, None]
                oq, _ = requant.requant_mxfp4_to_int4g32(w, np.array([[[s]]], np.uint8))
                nib = int(formats.unpack_nibbles(oq)[0, 0, 1])
                table.setdefault((cmax, c), set()).add(nib)
    assert all(len(v) == 1 for v in table.values())
    # spot values from the exact rule: code 7 (6.0) is the block max -> 7;
    # value 3 (code 5) under max 6 -> 7*3/6 = 3.5 decided by float32 rounding
    assert table[(7, 7)] == {7}
    assert table[(7, 15)] == {(-7) & 0xF}
    assert table[(7, 0)] == {0}


def test_requant_bf16_cast_is_identity_on_all_mxfp4_values():
    vals = formats.e2m1_decode(np.arange(16))[:, None] * formats.e8m0_decode(np.arange(255))[None, :]
    v32 = vals.astype(np.float32)
    finite = np.isfinite(v32)
    back = (formats.f32_to_bf16_rne(v32[finite]).astype(np.uint32) << 16).view(np.float32)
    assert np.array_equal(back, v32[finite])
    assert np.array_equal(v32[finite].astype(np.float64), vals[finite])


@pytest.mark.parametrize("chunk", [1, 3, 8, 100])
def test_requant_independent_of_chunk_size(chunk):
    g = np.random.default_rng(21)
    w = g.integers(0, 256, size=(10, 4, 32), dtype=np.uint8)
    sc = g.integers(110, 130, size=(10, 4, 2), dtype=np.uint8)
    a = requant.requant_mxfp4_to_int4g32(w, sc, 8)
    b = requant.requant_mxfp4_to_int4g32(w, sc, chunk)
    assert np.array_equal(a[0], b[0]) and np.array_equal(a[1].view(np.uint32), b[1].view(np.uint32))


def test_requant_never_reaches_minus_eight_and_reconstructs_max():
    g = np.random.default_rng(22)
    w = g.integers(0, 256, size=(3, 8, 64), dtype=np.uint8)
    sc = g.integers(110, 130, size=(3, 8, 4), dtype=np.uint8)
    q, s = requant.requant_mxfp4_to_int4g32(w, sc)
    codes = formats.unpack_nibbles(q).astype(np.int64)
    vals = np.where(codes >= 8, codes - 16, codes)
    assert vals.min() >= -7 and vals.max() <= 7
    deq = moe.dequant_int4(q, s)
    src = formats.dequant_mxfp4(w, sc)
    # error per element at most half a step (scale/2) plus float32 rounding of the scale
    step = np.repeat(s.astype(np.float64), 32, axis=-1)
    assert np.all(np.abs(deq - src) <= step * 0.5 * (1 + 1e-6) + 1e-30)


# ----------------------------------------------------------------------------- swiglu_limit clamp


def test_moe_swiglu_limit_matches_torch_clamp():
    x, ids, w, w13, s13, w2, s2 = _tiny_problem(61, T=6, topk=3)
    g = synth.rng(62)
    E, I2, H = w13.shape[0], w13.shape[1], w2.shape[1]
    b13 = _bias_bits(g, (E, I2), 2.0)
    X = torch.from_numpy(x.view(np.int16)).view(torch.bfloat16).double()
    W13 = torch.from_numpy(formats.dequant_mxfp4(w13, s13))
    W2 = torch.from_numpy(formats.dequant_mxfp4(w2, s2))
    B13 = torch.from_numpy(b13.view(np.int16)).view(torch.bfloat16).double()
    I = I2 // 2
    for limit in (0.3, 1.5):
        ours = moe.moe_forward(x, ids, w, w13, s13, w2, s2, b13=b13, swiglu_limit=limit)
        ref = torch.zeros(X.shape, dtype=torch.float64)
        for t in range(ids.shape[0]):
            for k in range(ids.shape[1]):
                e = int(ids[t, k])
                h = torch.clamp(torch.nn.functional.linear(X[t], W13[e], B13[e]), -limit, limit)
                a = torch.nn.functional.silu(h[:I]) * h[I:]
                ref[t] += float(w[t, k]) * torch.nn.functional.linear(a, W2[e])
        assert np.allclose(ours, ref.numpy(), rtol=1e-12, atol=1e-14)
        # the clamp is active: the result differs from the unclamped layer
        assert not np.allclose(ours, moe.moe_forward(x, ids, w, w13, s13, w2, s2, b13=b13), rtol=1e-3)


def test_moe_swiglu_limit_closed_forms():
    x, ids, w, w13, s13, w2, s2 = _tiny_problem(63, E=2, T=3, topk=1)
    base = moe.moe_forward(x, ids, w, w13, s13, w2, s2)
    # a limit above every |h| changes nothing
    assert np.array_equal(moe.moe_forward(x, ids, w, w13, s13, w2, s2, swiglu_limit=1e30), base)
    # all-zero gate_up codes: h is the bias alone, so the output is the clamped
    # bias pushed through SiLU gating and the down projection
    zero13 = np.zeros_like(w13)
    b13 = synth.bf16_bits_from_f32(np.full((2, w13.shape[1]), 3.0, np.float32))
    limit = 0.75
    out = moe.moe_forward(x, ids, w, zero13, s13, w2, s2, b13=b13, swiglu_limit=limit)
    I = w13.shape[1] // 2
    a = np.full(I, limit / (1.0 + np.exp(-limit)) * limit)
    W2 = formats.dequant_mxfp4(w2, s2)
    for t in range(3):
        e = ids[t, 0]
        assert np.allclose(out[t], float(np.float32(w[t, 0])) * (W2[e] @ a), rtol=1e-12)
