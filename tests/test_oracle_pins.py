"""Pins of the oracle against facts fixed outside it: hand-written fixtures,
closed forms, invariants, textbook routines and a dense brute force."""
import math
import os

import numpy as np
import pytest
import scipy.special

import oracle
from quantized_routed_expert_fn_gb300 import synth

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _golden_lines(name):
    with open(os.path.join(GOLDEN, name)) as f:
        for line in f:
            line = line.strip()
            if line and not line.startswith("#"):
                yield line


# ------------------------------------------------------------------ codes

def test_code_fixtures():
    n = 0
    for line in _golden_lines("codes.txt"):
        bits, words, codes = (p.strip() for p in line.split(";"))
        bits = int(bits)
        words = np.array([int(w, 16) for w in words.split()], dtype=np.uint32)
        codes = [int(c) for c in codes.split()]
        got = [oracle.code_at(words, i, bits) for i in range(len(codes))]
        assert got == codes, line
        n += 1
    assert n >= 6


def test_bf16_fixtures():
    for line in _golden_lines("bf16.txt"):
        b, v = line.split()
        assert oracle.bf16(int(b, 16)) == float(v)


@pytest.mark.parametrize("bits", [4, 3, 2])
def test_pack_unpack_every_code_every_position(bits):
    """Every code value at every position of a 64-code group survives the
    generator's packing and the oracle's unpacking."""
    n = 64
    vals = 1 << bits
    codes = np.array([[(i + r) % vals for i in range(n)] for r in range(vals)], dtype=np.uint32)
    words = synth.pack_codes(codes, bits)
    assert words.shape == (vals, n * bits // 32)
    for r in range(vals):
        got = [oracle.code_at(words[r], i, bits) for i in range(n)]
        assert got == list(codes[r])


@pytest.mark.parametrize("bits", [4, 3, 2])
def test_dequant_endpoints(bits):
    """Code 0 maps to the bias; the largest code to scale*(2^b-1) + bias."""
    lay = synth.record_layout(256, 64, bits)
    s_bits, b_bits = 0x3C00, 0xBD80  # 0.0078125, -0.0625
    s, b = 0.0078125, -0.0625
    for code, want in ((0, b), ((1 << bits) - 1, s * ((1 << bits) - 1) + b)):
        rec = synth.make_uniform_record(lay, code, s_bits, b_bits)[0]
        for q in (lay.gate_up, lay.down):
            W = oracle.dequant(rec, q, bits)
            assert W.shape == (q.out, q.inp)
            assert np.all(W == want)


def test_dequant_groups_are_64_wide():
    """A scale change at code 64 affects exactly codes 64..127 of a row."""
    lay = synth.record_layout(256, 64, 4)
    rec = synth.make_uniform_record(lay, 1, 0x3F80, 0x0000)[0].copy()
    q = lay.gate_up
    scales = rec[q.s:q.s + q.out * (q.inp // 64) * 2].view(np.uint16)
    scales[1] = 0x4000  # row 0, group 1 -> scale 2.0
    W = oracle.dequant(rec, q, 4)
    assert np.all(W[0, :64] == 1.0) and np.all(W[0, 64:128] == 2.0) and np.all(W[0, 128:] == 1.0)
    assert np.all(W[1:] == 1.0)


# ------------------------------------------------------------------ routing

def _sorted_topk(logits, k):
    order = sorted(range(len(logits)), key=lambda e: (-np.float32(logits[e]), e))
    return order[:k]


@pytest.mark.parametrize("E,k", [(8, 2), (128, 8), (512, 10), (16, 16), (5, 1)])
def test_topk_matches_full_sort(E, k):
    rng = np.random.default_rng(E * 31 + k)
    for _ in range(20):
        logits = rng.normal(0, 2, size=E)
        idx, w = oracle.topk_softmax(logits, k)
        assert list(idx) == _sorted_topk(logits, k)
        assert abs(w.sum() - 1.0) < 1e-12
        assert np.all(np.diff(w) <= 1e-15)


def test_topk_ties_lower_id_wins():
    logits = np.array([1.0, 3.0, 3.0, 2.0, 3.0, 0.5])
    idx, w = oracle.topk_softmax(logits, 3)
    assert list(idx) == [1, 2, 4]
    assert np.allclose(w, 1.0 / 3.0, atol=0, rtol=1e-15)


def test_softmax_reduces_to_textbook_when_k_is_e():
    rng = np.random.default_rng(3)
    logits = rng.normal(0, 3, size=40)
    idx, w = oracle.topk_softmax(logits, 40)
    ref = scipy.special.softmax(logits)
    assert np.allclose(w, ref[idx], rtol=1e-13, atol=0)


def test_softmax_shift_invariant_and_k1():
    rng = np.random.default_rng(4)
    logits = rng.normal(0, 1, size=64)
    i1, w1 = oracle.topk_softmax(logits, 6)
    i2, w2 = oracle.topk_softmax(logits + 17.0, 6)
    assert list(i1) == list(i2)
    assert np.allclose(w1, w2, rtol=1e-12, atol=0)
    i, w = oracle.topk_softmax(logits, 1)
    assert w[0] == 1.0 and i[0] == int(np.argmax(logits))


def test_union_first_seen_order():
    assert list(oracle.union(np.array([3, 1, 3, 2, 1, 7]))) == [3, 1, 2, 7]
    assert list(oracle.union(np.array([5, 5, 5]))) == [5]


# ------------------------------------------------------------------ expert math

def _uniform_layer(H, I, E, k, code, s_bits, b_bits, shared=False):
    lay = synth.record_layout(H, I, 4)
    rec = synth.make_uniform_record(lay, code, s_bits, b_bits)
    layer = synth.make_layer(np.random.default_rng(0), H, E, k, I, 4, shared=shared)
    layer.records = np.repeat(rec, E, axis=0)
    if shared:
        layer.shared_record = rec[0].copy()
    return layer


@pytest.mark.parametrize("H,I,E,k", [(64, 64, 2, 1), (256, 128, 8, 2)])
def test_closed_form_uniform_records(H, I, E, k):
    """All codes q, scale sigma, bias -8 sigma: every weight is c = sigma (q-8),
    so gate = up = c*S with S = sum(x), h = silu(cS)*cS and y = c*I*h for
    every output; routing weights sum to 1, so out = y."""
    sigma, q = 2.0 ** -6, 11
    layer = _uniform_layer(H, I, E, k, q, 0x3C80, 0xBE00)  # 0.015625, -0.125
    assert synth.bf16_bits_to_f32(np.array([0x3C80, 0xBE00], dtype=np.uint16)).tolist() == [sigma, -8 * sigma]
    c = sigma * (q - 8)
    x = np.random.default_rng(1).normal(size=(2, H))
    r = oracle.moe_layer(oracle.Layer(layer), x)
    for b in range(2):
        S = x[b].sum()
        g = c * S
        want = c * I * (g / (1 + math.exp(-g))) * g
        assert np.allclose(r["out"][b], want, rtol=1e-12, atol=1e-15)


def test_code_eight_with_bias_minus_eight_scale_gives_zero():
    layer = _uniform_layer(64, 64, 2, 1, 8, 0x3C80, 0xBE00)
    x = np.random.default_rng(2).normal(size=(1, 64))
    assert np.all(oracle.moe_layer(oracle.Layer(layer), x)["out"] == 0.0)


def test_zero_shared_gate_weights_half():
    """sigmoid(0) = 1/2: a zero shared-gate vector scales the shared expert by 0.5."""
    layer = synth.make_layer(np.random.default_rng(5), 128, 4, 1, 64, 4, shared=True)
    layer.shared_gate = np.zeros(128, dtype=np.uint16)
    ol = oracle.Layer(layer)
    x = np.random.default_rng(6).normal(size=(1, 128))
    r = oracle.moe_layer(ol, x)
    assert r["gamma"][0] == 0.5
    y_r = oracle.expert(ol, int(r["idx"][0, 0]), x[0])
    y_s = oracle.shared_expert(ol, x[0])
    assert np.allclose(r["out"][0], y_r + 0.5 * y_s, rtol=1e-13, atol=1e-15)


# ------------------------------------------------------------------ dense brute force

def _np_dequant(rec, q, bits):
    """Independent numpy decoding: expand each row's words to a bit array, then
    read `bits` consecutive bits per code, LSB first."""
    words = rec[q.w:q.w + q.out * q.inp * bits // 8].view("<u4").reshape(q.out, -1)
    shifts = np.arange(32, dtype=np.uint32)
    bitarr = ((words[:, :, None] >> shifts) & 1).reshape(q.out, -1)
    codes = bitarr.reshape(q.out, q.inp, bits) @ (1 << np.arange(bits))
    ng = q.inp // 64
    s = synth.bf16_bits_to_f32(rec[q.s:q.s + q.out * ng * 2].view(np.uint16)).astype(np.float64).reshape(q.out, ng)
    b = synth.bf16_bits_to_f32(rec[q.b:q.b + q.out * ng * 2].view(np.uint16)).astype(np.float64).reshape(q.out, ng)
    return np.repeat(s, 64, axis=1) * codes + np.repeat(b, 64, axis=1)


def _np_expert(rec, lay, bits, x):
    Wgu = _np_dequant(rec, lay.gate_up, bits)
    Wd = _np_dequant(rec, lay.down, bits)
    gu = Wgu @ x
    I = lay.inter
    h = gu[:I] * scipy.special.expit(gu[:I]) * gu[I:]
    return Wd @ h


@pytest.mark.parametrize("bits,shared,flags", [(4, False, 0), (4, True, 0), (3, True, 0), (2, True, 0),
                                               (4, True, synth.RESIDUAL | synth.PRENORM)])
def test_dense_bruteforce_all_experts_masked(bits, shared, flags):
    """Evaluate every expert densely, weight by the full softmax masked to the
    top-k and renormalised; must equal the oracle's routed evaluation."""
    H, E, k, I, nb = 128, 8, 3, 64, 3
    rng = np.random.default_rng(10 + bits)
    layer = synth.make_layer(rng, H, E, k, I, bits, shared=shared, flags=flags)
    x = rng.normal(size=(nb, H))
    r = oracle.moe_layer(oracle.Layer(layer), x)
    R = synth.bf16_bits_to_f32(layer.router).astype(np.float64)
    for b in range(nb):
        xb = x[b]
        if flags & synth.PRENORM:
            xb = xb / np.sqrt(np.mean(xb * xb) + 1e-6)
        logits = R @ xb
        p = scipy.special.softmax(logits)
        top = np.argsort(-logits, kind="stable")[:k]
        mask = np.zeros(E)
        mask[top] = 1
        wts = p * mask / (p * mask).sum()
        dense = sum(wts[e] * _np_expert(layer.records[e], layer.layout, bits, xb) for e in range(E))
        if shared:
            sg = synth.bf16_bits_to_f32(layer.shared_gate).astype(np.float64)
            dense = dense + scipy.special.expit(sg @ xb) * _np_expert(layer.shared_record, layer.shared_layout, 4, xb)
        if flags & synth.RESIDUAL:
            dense = dense + x[b]
        assert sorted(r["idx"][b]) == sorted(top)
        assert np.allclose(r["out"][b], dense, rtol=1e-9, atol=1e-12)


@pytest.mark.parametrize("flags", [0, synth.RESIDUAL | synth.PRENORM])
def test_mixed_width_dense_bruteforce(flags):
    """A union mixing 4-, 3- and 2-bit records: every expert evaluated densely
    at its own width by the independent numpy decoding, weighted by the
    masked, renormalised softmax; must equal the oracle's routed evaluation
    (which picks each record's width and offsets from the per-expert array)."""
    H, E, k, I, nb = 128, 12, 4, 64, 4
    rng = np.random.default_rng(31)
    eb = np.array([4, 3, 2] * 4, dtype=np.uint8)
    rng.shuffle(eb)
    layer = synth.make_mixed_layer(rng, H, E, k, I, eb, shared=True, flags=flags)
    x = rng.normal(size=(nb, H))
    r = oracle.moe_layer(oracle.Layer(layer), x)
    assert set(eb[r["union"]].tolist()) == {2, 3, 4}, "the union should hold every width"
    R = synth.bf16_bits_to_f32(layer.router).astype(np.float64)
    for b in range(nb):
        xb = x[b]
        if flags & synth.PRENORM:
            xb = xb / np.sqrt(np.mean(xb * xb) + 1e-6)
        logits = R @ xb
        p = scipy.special.softmax(logits)
        top = np.argsort(-logits, kind="stable")[:k]
        mask = np.zeros(E)
        mask[top] = 1
        wts = p * mask / (p * mask).sum()
        dense = sum(wts[e] * _np_expert(layer.records[e], layer.layouts[int(eb[e])], int(eb[e]), xb)
                    for e in range(E))
        sg = synth.bf16_bits_to_f32(layer.shared_gate).astype(np.float64)
        dense = dense + scipy.special.expit(sg @ xb) * _np_expert(layer.shared_record, layer.shared_layout, 4, xb)
        if flags & synth.RESIDUAL:
            dense = dense + x[b]
        assert sorted(r["idx"][b]) == sorted(top)
        assert np.allclose(r["out"][b], dense, rtol=1e-9, atol=1e-12)


def test_mixed_width_reads_each_record_at_its_own_width():
    """Reading a narrower record with the 4-bit layout gives a different
    expert: the per-expert widths are not a no-op."""
    H, E, k, I = 128, 6, 2, 64
    rng = np.random.default_rng(32)
    eb = np.array([4, 3, 2, 4, 3, 2], dtype=np.uint8)
    layer = synth.make_mixed_layer(rng, H, E, k, I, eb, shared=False)
    ol = oracle.Layer(layer)
    x = rng.normal(size=H)
    for e in range(E):
        b = int(eb[e])
        y = oracle.expert(ol, e, x)
        assert np.allclose(y, _np_expert(layer.records[e], layer.layouts[b], b, x), rtol=1e-9, atol=1e-12)
        if b != 4:
            assert not np.allclose(y, _np_expert(layer.records[e], layer.layouts[4], 4, x), rtol=1e-3)


# ------------------------------------------------------------------ tiers and the deadline cut

def _tiered(layer, tier, cut_w):
    import copy
    L = copy.copy(layer)
    L.expert_tier = np.ascontiguousarray(tier, dtype=np.uint8)
    L.cut_w = cut_w
    return L


def test_cut_rule_hand_example():
    """Two rows, top-2 of 6 experts.  Expert 3 (host memory) has weights 0.3
    and 0.05: kept, being above w = 0.2 in one row.  Expert 4 (host) has
    0.1 and 0.15: cut.  Expert 1 (device memory) has 0.05: never cut."""
    rng = np.random.default_rng(40)
    layer = synth.make_layer(rng, 128, 6, 2, 64, 4, shared=False)
    tier = np.array([0, 0, 1, 1, 1, 0], dtype=np.uint8)
    ol = oracle.Layer(_tiered(layer, tier, 0.2))
    idx = np.array([[3, 4], [1, 4]], dtype=np.int32)
    w = np.array([[0.3, 0.1], [0.05, 0.15]])
    assert oracle.cut(ol, idx, w).tolist() == [False, False, False, False, True, False]
    idx = np.array([[3, 1], [4, 1]], dtype=np.int32)
    w = np.array([[0.05, 0.95], [0.05, 0.95]])
    assert oracle.cut(ol, idx, w).tolist() == [False, False, False, True, True, False]
    assert not oracle.cut(oracle.Layer(_tiered(layer, tier, 0.0)), idx, w).any()


def test_cut_zero_threshold_changes_nothing():
    rng = np.random.default_rng(41)
    layer = synth.make_layer(rng, 128, 16, 4, 64, 4, shared=True, flags=synth.RESIDUAL | synth.PRENORM)
    x = rng.normal(size=(4, 128))
    base = oracle.moe_layer(oracle.Layer(layer), x)
    tiered = oracle.moe_layer(oracle.Layer(_tiered(layer, np.arange(16) % 2, 0.0)), x)
    assert np.array_equal(base["out"], tiered["out"])


def test_cut_of_every_host_expert_equals_zeroed_records():
    """With w above every possible weight, every host-memory expert is cut:
    the same as those experts' records being all zero (weight 0 everywhere,
    output 0), the routing unchanged."""
    rng = np.random.default_rng(42)
    layer = synth.make_layer(rng, 128, 16, 4, 64, 4, shared=True, flags=synth.PRENORM)
    tier = (np.arange(16) % 3 == 0).astype(np.uint8)
    x = rng.normal(size=(3, 128))
    cut = oracle.moe_layer(oracle.Layer(_tiered(layer, tier, 1.0)), x)
    import copy
    z = copy.copy(layer)
    z.records = layer.records.copy()
    z.records[tier == 1] = 0
    ref = oracle.moe_layer(oracle.Layer(z), x)
    assert np.array_equal(cut["idx"], ref["idx"])
    assert np.allclose(cut["out"], ref["out"], rtol=0, atol=1e-13)


def test_cut_dense_bruteforce():
    """Threshold in the middle of the routed weights: every expert densely,
    each host-memory expert dropped when its max weight over the rows is
    below w, others weighted as usual."""
    H, E, k, I, nb = 128, 16, 4, 64, 4
    rng = np.random.default_rng(43)
    layer = synth.make_layer(rng, H, E, k, I, 4, shared=True)
    tier = (rng.random(E) < 0.5).astype(np.uint8)
    x = rng.normal(size=(nb, H))
    R = synth.bf16_bits_to_f32(layer.router).astype(np.float64)
    W = np.zeros((nb, E))
    for b in range(nb):
        logits = R @ x[b]
        top = np.argsort(-logits, kind="stable")[:k]
        p = scipy.special.softmax(logits[top])
        W[b, top] = p
    w_cut = float(np.median(W[W > 0]))
    r = oracle.moe_layer(oracle.Layer(_tiered(layer, tier, w_cut)), x)
    dropped = (tier == 1) & (W.max(axis=0) > 0) & (W.max(axis=0) < w_cut)
    assert dropped.any() and ((tier == 1) & (W.max(axis=0) >= w_cut)).any()
    sg = synth.bf16_bits_to_f32(layer.shared_gate).astype(np.float64)
    for b in range(nb):
        dense = sum(W[b, e] * _np_expert(layer.records[e], layer.layout, 4, x[b]) for e in range(E) if not dropped[e])
        dense = dense + scipy.special.expit(sg @ x[b]) * _np_expert(layer.shared_record, layer.shared_layout, 4, x[b])
        assert np.allclose(r["out"][b], dense, rtol=1e-9, atol=1e-12)


def test_batch_rows_are_independent():
    rng = np.random.default_rng(20)
    layer = oracle.Layer(synth.make_layer(rng, 128, 8, 2, 64, 4))
    x = rng.normal(size=(4, 128))
    r4 = oracle.moe_layer(layer, x)
    for b in range(4):
        r1 = oracle.moe_layer(layer, x[b:b + 1])
        assert np.array_equal(r1["out"][0], r4["out"][b])
        assert list(r1["idx"][0]) == list(r4["idx"][b])


def test_expert_relabeling_leaves_output_unchanged():
    rng = np.random.default_rng(21)
    src = synth.make_layer(rng, 128, 8, 2, 64, 4)
    x = rng.normal(size=(2, 128))
    r = oracle.moe_layer(oracle.Layer(src), x)
    perm = rng.permutation(8)
    src.router = src.router[perm].copy()
    src.records = src.records[perm].copy()
    rp = oracle.moe_layer(oracle.Layer(src), x)
    assert np.allclose(r["out"], rp["out"], rtol=1e-12, atol=1e-15)
    assert sorted(perm[rp["idx"][0]]) == sorted(r["idx"][0])


def test_union_and_wmap_consistent():
    rng = np.random.default_rng(22)
    layer = oracle.Layer(synth.make_layer(rng, 128, 16, 4, 64, 4))
    x = rng.normal(size=(4, 128))
    r = oracle.moe_layer(layer, x)
    U = r["union"]
    assert len(set(U.tolist())) == len(U) == len(set(r["idx"].reshape(-1).tolist()))
    for b in range(4):
        assert abs(r["wmap"][b, :len(U)].sum() - 1.0) < 1e-12
        for j, e in enumerate(U):
            want = r["w"][b][list(r["idx"][b]).index(e)] if e in r["idx"][b] else 0.0
            assert r["wmap"][b, j] == want


def test_stacked_layers_compose():
    rng = np.random.default_rng(23)
    layers = [synth.make_layer(rng, 128, 8, 2, 64, 4, flags=synth.RESIDUAL | synth.PRENORM) for _ in range(3)]
    ol = [oracle.Layer(l) for l in layers]
    x = rng.normal(size=(2, 128))
    f = oracle.moe_forward(ol, x)
    cur = x
    for l in range(3):
        assert np.array_equal(f["inputs"][l], cur)
        cur = oracle.moe_layer(ol[l], cur)["out"]
    assert np.array_equal(f["out"], cur)


def test_prenorm_is_scale_invariant():
    rng = np.random.default_rng(24)
    layer = oracle.Layer(synth.make_layer(rng, 128, 8, 2, 64, 4, flags=synth.PRENORM))
    x = rng.normal(size=(1, 128))
    a = oracle.moe_layer(layer, x)["out"]
    b = oracle.moe_layer(layer, 4.0 * x)["out"]
    # rmsnorm(4x) differs from rmsnorm(x) only through eps = 1e-6 (relative ~1e-6)
    assert np.abs(a - b).max() <= 1e-5 * np.abs(a).max()


def test_prefill_rows_match_layer_and_mirror_is_bf16():
    rng = np.random.default_rng(25)
    layer = synth.make_layer(rng, 128, 16, 4, 64, 4)
    ol = oracle.Layer(layer)
    x = rng.normal(size=(6, 128)).astype(np.float32)
    rows = np.array([0, 3, 5])
    exact = oracle.prefill_rows(ol, x, rows, mirror=False)
    mir = oracle.prefill_rows(ol, x, rows, mirror=True)
    ref = oracle.moe_layer(ol, x[rows].astype(np.float64))
    assert np.allclose(exact["out"], ref["out"], rtol=1e-13, atol=1e-15)
    assert np.array_equal(exact["idx"], ref["idx"])
    rms = np.sqrt((exact["out"] ** 2).mean(axis=1, keepdims=True))
    assert np.all(np.abs(mir["out"] - exact["out"]) < 3e-2 * rms)
    m32 = mir["out"].astype(np.float32)
    assert np.array_equal(m32.view(np.uint32) & 0xFFFF, np.zeros_like(m32, dtype=np.uint32))


# ------------------------------------------------------------------ prefill routing and grouping

def _np_rmsnorm(x):
    return x / np.sqrt((x * x).mean(axis=1, keepdims=True) + 1e-6)


@pytest.mark.parametrize("flags", [0, synth.PRENORM])
def test_route_rows_match_numpy_bruteforce(flags):
    rng = np.random.default_rng(31)
    layer = synth.make_layer(rng, 256, 24, 5, 64, 4, flags=flags)
    ol = oracle.Layer(layer)
    x = rng.normal(size=(40, 256)).astype(np.float32)
    r = oracle.route_rows(ol, x)
    xh = x.astype(np.float64)
    if flags & synth.PRENORM:
        xh = _np_rmsnorm(xh)
    R = synth.bf16_bits_to_f32(layer.router).astype(np.float64)
    logits = xh @ R.T
    assert np.allclose(r["logits"], logits, rtol=1e-12, atol=1e-12)
    for b in range(x.shape[0]):
        order = np.lexsort((np.arange(24), -logits[b].astype(np.float32)))[:5]
        assert r["idx"][b].tolist() == order.tolist()
        assert np.allclose(r["w"][b], scipy.special.softmax(logits[b][order]), rtol=1e-12, atol=0)
    sg = synth.bf16_bits_to_f32(layer.shared_gate).astype(np.float64)
    assert np.allclose(r["gamma"], scipy.special.expit(xh @ sg), rtol=1e-12, atol=0)


def test_group_hand_example():
    # 4 rows, 3 experts, k = 2; worked by hand:
    #   row 0 -> {2, 0}, row 1 -> {0, 1}, row 2 -> {2, 1}, row 3 -> {1, 0}
    #   expert 0: rows 0, 1, 3; expert 1: rows 1, 2, 3; expert 2: rows 0, 2;
    #   shared group: rows 0..3
    idx = np.array([[2, 0], [0, 1], [2, 1], [1, 0]])
    w = np.array([[0.6, 0.4], [0.7, 0.3], [0.55, 0.45], [0.9, 0.1]])
    gamma = np.array([0.1, 0.2, 0.3, 0.4])
    g = oracle.group(3, idx, w, gamma)
    assert g["offs"].tolist() == [0, 3, 6, 8, 12]
    assert g["rows"].tolist() == [0, 1, 3, 1, 2, 3, 0, 2, 0, 1, 2, 3]
    assert g["wts"].tolist() == [0.4, 0.7, 0.1, 0.3, 0.45, 0.9, 0.6, 0.55, 0.1, 0.2, 0.3, 0.4]
    g2 = oracle.group(3, idx, w, None)
    assert g2["offs"].tolist() == [0, 3, 6, 8]
    assert g2["rows"].tolist() == [0, 1, 3, 1, 2, 3, 0, 2]


def test_group_invariants_random():
    rng = np.random.default_rng(32)
    n, E, k = 300, 37, 6
    idx = np.stack([rng.choice(E, size=k, replace=False) for _ in range(n)]).astype(np.int32)
    w = rng.random((n, k))
    g = oracle.group(E, idx, w, None)
    offs, rows, wts = g["offs"], g["rows"], g["wts"]
    assert np.array_equal(np.diff(offs), np.bincount(idx.ravel(), minlength=E))
    seen = set()
    for e in range(E):
        rs = rows[offs[e]:offs[e + 1]]
        assert np.all(np.diff(rs) > 0), "rows ascend inside a group"
        for p, r in zip(range(offs[e], offs[e + 1]), rs):
            j = int(np.nonzero(idx[r] == e)[0][0])
            assert wts[p] == w[r, j]
            seen.add((int(r), e))
    assert len(seen) == n * k


@pytest.mark.parametrize("bits", [4, 3, 2])
def test_prefill_mirror_matches_dense_bf16_bruteforce(bits):
    """The bf16 mirror equals a dense numpy evaluation with x^, W, h and the
    output rounded to bf16 (round to nearest even, via float32, exact here);
    routed records of every width, the shared record 4-bit."""
    rng = np.random.default_rng(33 + bits)
    H, E, k, I = 128, 6, 2, 64
    layer = synth.make_layer(rng, H, E, k, I, bits, flags=synth.RESIDUAL | synth.PRENORM)
    ol = oracle.Layer(layer)
    x = rng.normal(size=(5, H)).astype(np.float32)
    got = oracle.prefill_rows(ol, x, np.arange(5), mirror=True)

    def bf(a):
        return synth.bf16_bits_to_f32(synth.f32_to_bf16_bits(np.asarray(a, dtype=np.float32))).astype(np.float64)

    def dense(rec, lay, bits):
        return bf(oracle.dequant(rec, lay.gate_up, bits)), bf(oracle.dequant(rec, lay.down, bits))

    xh = _np_rmsnorm(x.astype(np.float64))
    xe = bf(xh)
    R = synth.bf16_bits_to_f32(layer.router).astype(np.float64)
    sg = synth.bf16_bits_to_f32(layer.shared_gate).astype(np.float64)
    for b in range(5):
        lg = R @ xh[b]
        ids = np.lexsort((np.arange(E), -lg.astype(np.float32)))[:k]
        wt = scipy.special.softmax(lg[ids])
        acc = np.zeros(H)
        experts = [(layer.records[e], layer.layout, layer.bits, wt[j]) for j, e in enumerate(ids)]
        experts.append((layer.shared_record, layer.shared_layout, 4, scipy.special.expit(sg @ xh[b])))
        for rec, lay, bits, wgt in experts:
            Wgu, Wd = dense(rec, lay, bits)
            gu = Wgu @ xe[b]
            h = bf(gu[:I] / (1.0 + np.exp(-gu[:I])) * gu[I:])
            acc += wgt * (Wd @ h)
        want = bf(acc + x[b])
        ulp = np.abs(want) * 2.0 ** -7
        assert np.all(np.abs(got["out"][b] - want) <= ulp), f"row {b}"
        assert np.mean(got["out"][b] == want) > 0.99


# ------------------------------------------------------------------ bf16 mirror helpers

def test_round_bf16_fixtures():
    """The mirror's bf16 rounding against hand-written round-to-nearest-even
    cases: exact ties both ways, values just off a tie, negatives, a carry
    into the exponent."""
    n = 0
    for line in _golden_lines("bf16_round.txt"):
        v, b = line.split()
        got = oracle.round_bf16(float(v))
        want = oracle.bf16(int(b, 16))
        assert got == want, f"{v}: {got!r} != {want!r} (bits {b})"
        n += 1
    assert n >= 12


def _allowance_record(q63: int):
    """A hand-built 4-bit expert, hidden 64, inter 64 (one 64-code group per row):
      gate row 0: scale 0.5, codes (2, 1 x 62, 0)       -> g0 = 32 on the x below
      up row 0:   scale 2^-14, codes 15 x 34, 1, 0 ..., q63 at position 63
                                                      -> u0 = 2^-14 (511 + q63 2^-11)
      every other up row: scale 0 -> u = 0, h = 0 (never near a boundary)
      down: fixed bf16 weights, W_d[o][0] = (o + 1) / 64 (scale 1/64, code o % 15 + 1)
    with x = (1 x 63, 2^-11).  Then h0 = silu(32) u0 = 511/512 + q63 2^-20 (up to
    a relative 1.3e-14): just above the bf16 midpoint 0.998046875 between
    0.99609375 and 1.0, so h0 rounds to 1.0 and the value across the boundary
    is 0.99609375 (one step of 2^-8 below)."""
    lay = synth.record_layout(64, 64, 4)
    rec = np.zeros(lay.stride, dtype=np.uint8)
    gu, dn = lay.gate_up, lay.down
    codes = np.zeros((128, 64), dtype=np.uint32)
    codes[0, 0], codes[0, 1:63] = 2, 1
    codes[64, :34], codes[64, 34], codes[64, 63] = 15, 1, q63
    rec[gu.w:gu.w + 128 * 32] = synth.pack_codes(codes, 4).reshape(-1).view(np.uint8)
    s = np.zeros(128, dtype=np.uint16)
    s[0], s[64] = 0x3F00, 0x3880  # 0.5, 2^-14
    rec[gu.s:gu.s + 256] = s.view(np.uint8)
    dcodes = np.zeros((64, 64), dtype=np.uint32)
    dcodes[:, 0] = np.arange(64) % 15 + 1
    dcodes[:, 1:] = 3
    rec[dn.w:dn.w + 64 * 32] = synth.pack_codes(dcodes, 4).reshape(-1).view(np.uint8)
    rec[dn.s:dn.s + 128] = np.full(64, 0x3C80, dtype=np.uint16).view(np.uint8)  # 1/64
    x = np.ones(64)
    x[63] = 2.0 ** -11
    return rec, lay, x, (dcodes[:, 0] / 64.0)


def test_flip_allowance_hand_case():
    """The allowance that widens the prefill bound, pinned by hand.  The band
    of h0 is 2^-20 (|silu(g)| sum|up terms| + 1.1 |u| sum|gate terms|) +
    2^-22 |h| ~= 2^-20 (0.998 + 1.098) + 2.4e-7 ~= 2.24e-6.
      q63 = 2: h0 sits 2 x 2^-20 = 1.9e-6 above the midpoint -> inside the band:
               allow[o] = |w W_d[o][0] (0.99609375 - 1.0)| = |w W_d[o][0]| 2^-8 exactly;
      q63 = 3: 3 x 2^-20 = 2.9e-6 above it -> outside: allow = 0.
    A band exponent one off either way (-19 or -21), a truncating bf16 round,
    or the neighbour taken on the wrong side each breaks one of the two."""
    w = 0.75
    rec, lay, x, wd0 = _allowance_record(2)
    assert oracle.round_bf16(0.998046875 + 2 * 2.0 ** -20) == 1.0
    r = oracle.expert_mirror(rec, lay, x, w)
    np.testing.assert_array_equal(r["allow"], np.abs(w * wd0) * 2.0 ** -8)
    rec, lay, x, _ = _allowance_record(3)
    r = oracle.expert_mirror(rec, lay, x, w)
    assert np.all(r["allow"] == 0.0)


def test_flip_allowance_zero_far_from_boundaries():
    """h exactly on a bf16 value far from any midpoint (h0 = 1.0 - 1.3e-14 with
    up codes summing to 512) carries no allowance."""
    rec, lay, x, _ = _allowance_record(0)
    codes = np.zeros((128, 64), dtype=np.uint32)
    codes[0, 0], codes[0, 1:63] = 2, 1
    codes[64, :34], codes[64, 34], codes[64, 35] = 15, 1, 1  # sum 512 -> h0 = silu(32)/32 ~ 1.0
    gu = lay.gate_up
    rec[gu.w:gu.w + 128 * 32] = synth.pack_codes(codes, 4).reshape(-1).view(np.uint8)
    r = oracle.expert_mirror(rec, lay, x, 1.0)
    assert np.all(r["allow"] == 0.0)
