"""GPU parity of the prefill chunk path (moe_prefill, moe_prefill_group) against the oracle.

Outputs are bf16, so they are graded against the oracle's bf16 mirror (x^, the
dequantized weights, h and the output rounded to bf16 where the tensor-core
path stores bf16): |gpu - oracle| <= 2e-3 * RMS(MoE row) + 1 bf16 ulp of the
oracle element + the oracle's one-flip allowance.  The allowance covers an h
whose exact value sits within fp32 accumulation accuracy of a bf16 rounding
boundary, so that a kernel summing in fp32 may round it to the other side;
one such flip moves the output by |w * W_d[o][i] * (bf16 step of h_i)|, and
the allowance is the largest such move among the row's ambiguous h.
Routing ids are exact where the k-th and (k+1)-th logits differ by at least
1e-3; the grouping is exact (it is a function of the ids).
"""
import numpy as np
import pytest

import oracle
from helpers import GAP, TOL, topk_gap
from quantized_routed_expert_fn_gb300 import synth

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def moe():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from quantized_routed_expert_fn_gb300 import build, moe as m
    build.build()
    m.lib()
    return m


def bf16_ulp(v: np.ndarray) -> np.ndarray:
    _, e = np.frexp(np.abs(v))  # |v| = f * 2^e, f in [0.5, 1)
    return np.ldexp(1.0, e - 8)


def gaps_of(logits, k):
    return np.array([topk_gap(logits[b], k) for b in range(logits.shape[0])])


def rows_with_gap(ol, rng, t, H, zipf=False):
    """t rows (seeded) whose top-k gap is >= GAP; rows are independent, so
    rows without the gap are dropped and replaced."""
    k = ol.src.top_k
    keep = []
    while sum(len(a) for a in keep) < t:
        x = synth.make_prefill_x(rng, t, H) if zipf else rng.normal(size=(t, H)).astype(np.float32)
        g = gaps_of(oracle.route_rows(ol, x)["logits"], k)
        keep.append(x[g >= GAP])
    return np.ascontiguousarray(np.concatenate(keep)[:t])


def run_prefill(m, dl, x):
    t, H = x.shape
    k = dl.src[0].top_k
    xt = torch.from_numpy(np.ascontiguousarray(x, dtype=np.float32)).cuda()
    out = torch.empty((t, H), dtype=torch.int16, device="cuda")
    idx = torch.zeros((t, k), dtype=torch.int32, device="cuda")
    ws = m.alloc_workspace(m.prefill_workspace(dl, t))
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    m.prefill(dl, xt, out, ws, status, idx)
    torch.cuda.synchronize()
    assert status.item() == 0, m.STATUS_NAMES.get(status.item())
    o = synth.bf16_bits_to_f32(out.cpu().numpy().view(np.uint16)).astype(np.float64)
    return o, idx.cpu().numpy()


def run_group(m, dl, x):
    t, H = x.shape
    L = dl.src[0]
    k, E = L.top_k, L.n_experts
    shared = L.shared_gate is not None
    G = E + (1 if shared else 0)
    ent = t * k + (t if shared else 0)
    xt = torch.from_numpy(np.ascontiguousarray(x, dtype=np.float32)).cuda()
    idx = torch.zeros((t, k), dtype=torch.int32, device="cuda")
    w = torch.zeros((t, k), dtype=torch.float32, device="cuda")
    offs = torch.full((G + 1,), -1, dtype=torch.int32, device="cuda")
    rows = torch.full((ent,), -1, dtype=torch.int32, device="cuda")
    wts = torch.zeros((ent,), dtype=torch.float32, device="cuda")
    ws = m.alloc_workspace(m.prefill_workspace(dl, t))
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    m.prefill_group(dl, xt, idx, w, offs, rows, wts, ws, status)
    torch.cuda.synchronize()
    assert status.item() == 0, m.STATUS_NAMES.get(status.item())
    return {k_: v.cpu().numpy() for k_, v in dict(idx=idx, w=w, offs=offs, rows=rows, wts=wts).items()}


def moe_rms(ref_out, x, flags):
    moe_part = ref_out - (x.astype(np.float64) if flags & synth.RESIDUAL else 0.0)
    return np.sqrt((moe_part ** 2).mean(axis=1))


def assert_prefill_close(got, ref, x, flags, rows, what):
    out, allow = ref["out"], ref["allow"]
    rms = moe_rms(out, x[rows], flags)
    base = TOL * rms[:, None] + bf16_ulp(out)
    bound = base + allow
    err = np.abs(got - out)
    bad = err > bound
    assert not bad.any(), f"{what}: {bad.sum()} elements over the bound, worst row {np.argmax(bad.any(axis=1))}"
    r = float((err / bound).max())
    n_base = int((err > base).sum())
    print(f"[parity] {what}: max err = {r:.4f} of the bound (2e-3 x row RMS + 1 bf16 ulp + flip allowance); "
          f"{n_base} of {err.size} elements need the allowance; mean allowance {float((allow / rms[:, None]).mean()):.2e} x RMS")
    return r


SMALL = [
    # H, E, k, I, t, shared, flags
    (256, 8, 2, 128, 1, False, 0),
    (256, 8, 2, 128, 37, True, 0),
    (768, 40, 5, 384, 300, True, synth.RESIDUAL | synth.PRENORM),
    (512, 130, 4, 192, 129, True, synth.PRENORM),
    (256, 4, 4, 64, 600, False, synth.RESIDUAL),
    (256, 16, 1, 128, 70, True, synth.PRENORM),  # top_k = 1
    (256, 1024, 4, 64, 50, True, 0),  # the most experts: most groups empty
    (256, 64, 32, 64, 40, False, 0),  # the largest top_k
    (256, 1, 1, 64, 33, True, 0),  # a single expert: every row routes to it, weight 1
]


@pytest.mark.parametrize("H,E,k,I,t,shared,flags", SMALL)
def test_prefill_small(moe, H, E, k, I, t, shared, flags):
    """Several token tiles with a ragged tail, expert groups above the 256-token
    tile, a router tile with padded experts, k == E, t == 1, k == 1, the most
    experts (1024) and the largest k (32)."""
    rng = np.random.default_rng(1000 + H + E + t)
    layer = synth.make_layer(rng, H, E, k, I, 4, shared=shared, flags=flags)
    ol = oracle.Layer(layer)
    x = rows_with_gap(ol, rng, t, H)
    dl = moe.DeviceLayers([layer])
    got, idx = run_prefill(moe, dl, x)
    ref = oracle.prefill_rows(ol, x, np.arange(t), mirror=True)
    assert np.array_equal(idx, ref["idx"]), "top-k ids"
    assert_prefill_close(got, ref, x, flags, np.arange(t), f"prefill H{H} E{E} k{k} I{I} t{t}")


@pytest.mark.parametrize("H,E,k,I,t,shared,flags", SMALL)
def test_prefill_group_small(moe, H, E, k, I, t, shared, flags):
    rng = np.random.default_rng(2000 + H + E + t)
    layer = synth.make_layer(rng, H, E, k, I, 4, shared=shared, flags=flags)
    ol = oracle.Layer(layer)
    x = rows_with_gap(ol, rng, t, H)
    g = run_group(moe, moe.DeviceLayers([layer]), x)
    r = oracle.route_rows(ol, x)
    assert np.array_equal(g["idx"], r["idx"])
    # the router reads x^ as two bf16 terms (relative error <= 2^-16), so
    # weights agree to about 1e-6; 1e-5 as in the decode routing tests
    assert np.allclose(g["w"], r["w"], rtol=0, atol=1e-5)
    ref = oracle.group(E, r["idx"], r["w"], r["gamma"])
    assert np.array_equal(g["offs"], ref["offs"]), "group offsets"
    assert np.array_equal(g["rows"], ref["rows"]), "grouped rows (stable order)"
    assert np.allclose(g["wts"], ref["wts"], rtol=0, atol=1e-5), "grouped weights"


LOWBIT = [
    # H, E, k, I, t, shared, flags, bits
    (768, 40, 5, 384, 300, True, synth.RESIDUAL | synth.PRENORM, 3),
    (512, 130, 4, 256, 129, True, synth.PRENORM, 3),
    (768, 40, 5, 384, 300, True, synth.RESIDUAL | synth.PRENORM, 2),
    (256, 8, 2, 192, 37, False, 0, 2),
]


@pytest.mark.parametrize("H,E,k,I,t,shared,flags,bits", LOWBIT)
def test_prefill_lowbit(moe, H, E, k, I, t, shared, flags, bits):
    """2- and 3-bit routed records (the shared expert stays 4-bit): codes that
    straddle 32-bit words, rows of 16 or 24 bytes a k-panel."""
    rng = np.random.default_rng(3000 + H + E + t + bits)
    layer = synth.make_layer(rng, H, E, k, I, bits, shared=shared, flags=flags, scale=(0.01, 0.04), bias_noise=0.0)
    ol = oracle.Layer(layer)
    x = rows_with_gap(ol, rng, t, H)
    dl = moe.DeviceLayers([layer])
    got, idx = run_prefill(moe, dl, x)
    ref = oracle.prefill_rows(ol, x, np.arange(t), mirror=True)
    assert np.array_equal(idx, ref["idx"]), "top-k ids"
    assert_prefill_close(got, ref, x, flags, np.arange(t), f"prefill {bits}-bit H{H} E{E} k{k} I{I} t{t}")


def test_prefill_rejects_unaligned_3bit_rows(moe):
    # 3-bit rows of inter 192 codes are 72 bytes: not a multiple of 16
    rng = np.random.default_rng(5)
    layer = synth.make_layer(rng, 256, 8, 2, 192, 3, shared=False)
    dl = moe.DeviceLayers([layer])
    assert moe.prefill_workspace(dl, 16) == 0
    x = torch.zeros((16, 256), dtype=torch.float32, device="cuda")
    out = torch.empty((16, 256), dtype=torch.int16, device="cuda")
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    ws = moe.alloc_workspace(1 << 20)
    with pytest.raises(moe.MoeError) as e:
        moe.prefill(dl, x, out, ws, status)
    assert e.value.code == moe.ESHAPE


def full_size_chunk(workload, t=4096):
    """The 4096-token prefill chunk: hidden 2048, 512 experts, top-10, inter 512,
    shared expert, Zipf(1.1) expert popularity through the router's bias channel."""
    rng = np.random.default_rng(4)
    layer = synth.make_config_layers(workload, seed=4)[0]
    synth.zipf_router(rng, layer)
    x = synth.make_prefill_x(rng, t, layer.hidden)
    return layer, oracle.Layer(layer), x


@pytest.fixture(scope="module")
def c4():
    return full_size_chunk("c4")


@pytest.fixture(scope="module")
def c4b3():
    return full_size_chunk("c4b3")


TILE_N = 160  # token columns of one tensor-core tile of the grouped GEMMs


def sampled_rows(ids, same, n_min=512, seed=44):
    """Rows to grade at full size: the first and last rows; one row in every
    token tile of the largest expert group (its rows in group order are the
    routed rows in token order); a row routed to each of the 64 rarest used
    experts; random rows up to n_min.  Only rows whose GPU id set equals the
    oracle's are kept (their outputs are comparable)."""
    t = ids.shape[0]
    counts = np.bincount(ids.ravel())
    members = np.nonzero((ids == int(np.argmax(counts))).any(axis=1))[0]
    tiles = members[::TILE_N].tolist() + [int(members[-1])]
    used = [int(e) for e in np.argsort(counts, kind="stable") if counts[e] > 0][:64]
    rare = [int(np.nonzero((ids == e).any(axis=1))[0][0]) for e in used]
    pick = set([0, t - 1] + tiles + rare)
    srng = np.random.default_rng(seed)
    for b in srng.permutation(t):
        if len([r for r in pick if same[r]]) >= n_min:
            break
        pick.add(int(b))
    rows = np.array(sorted(r for r in pick if same[r]))
    return rows, dict(tiles=len(tiles), rare=len(rare), largest=int(counts.max()))


def check_full_size(moe, chunk, what, n_min=512):
    layer, ol, x = chunk
    t, k, E = x.shape[0], layer.top_k, layer.n_experts
    dl = moe.DeviceLayers([layer])
    got, idx = run_prefill(moe, dl, x)
    r = oracle.route_rows(ol, x)
    gaps = gaps_of(r["logits"], k)
    clear = gaps >= GAP
    # rows with a clear top-k: the same chosen experts, in the oracle's order
    # except between chosen experts whose logits agree within the logit
    # tolerance the route test grants the kernels (1e-4 x the row's largest
    # |logit|): their order is not unique between two computations; near
    # ties: the first k-1 ids agree and the k-th is an expert whose logit is
    # within GAP of the oracle's k-th
    assert np.array_equal(np.sort(idx[clear], axis=1), np.sort(r["idx"][clear], axis=1))
    swaps = 0
    for b in np.nonzero(clear & np.any(idx != r["idx"], axis=1))[0]:
        seq = r["logits"][b][idx[b]]
        tol = 1e-4 * np.abs(r["logits"][b]).max()
        assert np.all(seq[1:] <= seq[:-1] + tol), (b, idx[b], r["idx"][b])
        swaps += 1
    for b in np.nonzero(~clear)[0]:
        assert sorted(idx[b][:k - 1]) == sorted(r["idx"][b][:k - 1])
        kth = np.sort(r["logits"][b].astype(np.float32))[::-1][k - 1]
        assert abs(float(r["logits"][b][idx[b][k - 1]]) - float(kth)) < GAP
    same = np.array([sorted(idx[b]) == sorted(r["idx"][b]) for b in range(t)])
    counts = np.bincount(r["idx"].ravel(), minlength=E)
    print(f"[{what}] rows with a top-k gap < {GAP}: {int((~clear).sum())}; id sets differing: {int((~same).sum())}; "
          f"rows ordering two chosen experts within the logit tolerance the other way: {swaps}; "
          f"expert rows max {counts.max()} min {counts.min()} empty {(counts == 0).sum()}")
    rows, info = sampled_rows(r["idx"], same, n_min=n_min)
    assert len(rows) >= n_min
    ref = oracle.prefill_rows(ol, x, rows, mirror=True)
    assert_prefill_close(got[rows], ref, x, layer.flags, rows,
                         f"{what} t={t} ({len(rows)} rows: {info['tiles']} tiles of the largest group of "
                         f"{info['largest']}, {info['rare']} rarest experts)")
    # reported, not graded: the distance from the exact (unrounded) oracle
    exact = oracle.prefill_rows(ol, x, rows, mirror=False)
    rms = moe_rms(exact["out"], x[rows], layer.flags)
    rel = np.abs(got[rows] - exact["out"]) / rms[:, None]
    print(f"[{what}] against the exact oracle (no bf16 rounding): max |err| = {rel.max():.3e} x row RMS, "
          f"mean {rel.mean():.3e} x row RMS")


def test_prefill_c4_full_size(moe, c4):
    check_full_size(moe, c4, "c4")


def test_prefill_c4b3_full_size(moe, c4b3):
    """The same chunk over 3-bit routed records (the shared expert stays 4-bit)."""
    check_full_size(moe, c4b3, "c4b3")


def test_prefill_large_chunk(moe):
    """A chunk 16 times the 4096-token one (65536 rows, the same layer): 2048
    grouping chunks, a shared-expert group of 65536 entries and the most
    popular expert in ~400 token tiles.  Every row's ids against the oracle;
    outputs on sampled rows, one in every token tile of the largest group."""
    check_full_size(moe, full_size_chunk("c4", t=65536), "c4 x16", n_min=256)


def test_prefill_bounded_wait_reports_timeout(moe):
    """A pipeline stage of the gate_up GEMM that never completes: every wait
    behind it gives up within the limit, the call reports MOE_ETIMEOUT, and
    the next call on the same context is correct."""
    import os
    rng = np.random.default_rng(301)
    H, E, k, I, t = 256, 8, 2, 128, 64
    layer = synth.make_layer(rng, H, E, k, I, 4, shared=True)
    ol = oracle.Layer(layer)
    x = rows_with_gap(ol, rng, t, H)
    dl = moe.DeviceLayers([layer])
    dl.set_flags(moe.TEST_WITHHOLD)
    xt = torch.from_numpy(x).cuda()
    out = torch.empty((t, H), dtype=torch.int16, device="cuda")
    ws = moe.alloc_workspace(moe.prefill_workspace(dl, t))
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    old = os.environ.get("MOE_TIMEOUT_MS")
    os.environ["MOE_TIMEOUT_MS"] = "50"
    try:
        moe.prefill(dl, xt, out, ws, status)
        torch.cuda.synchronize()
    finally:
        if old is None:
            del os.environ["MOE_TIMEOUT_MS"]
        else:
            os.environ["MOE_TIMEOUT_MS"] = old
    assert status.item() == moe.ETIMEOUT, moe.STATUS_NAMES.get(status.item())
    dl.set_flags(0)
    got, idx = run_prefill(moe, dl, x)
    ref = oracle.prefill_rows(ol, x, np.arange(t), mirror=True)
    assert np.array_equal(idx, ref["idx"])
    assert_prefill_close(got, ref, x, 0, np.arange(t), "prefill after a timed-out call")


def test_prefill_c4_group(moe, c4):
    """Full-size grouping: exactly the oracle's grouping of the GPU's own ids."""
    layer, ol, x = c4
    g = run_group(moe, moe.DeviceLayers([layer]), x)
    r = oracle.route_rows(ol, x)
    ref = oracle.group(layer.n_experts, g["idx"], g["w"].astype(np.float64), r["gamma"])
    assert np.array_equal(g["offs"], ref["offs"])
    assert np.array_equal(g["rows"], ref["rows"])
    assert np.allclose(g["wts"][:-x.shape[0]], ref["wts"][:-x.shape[0]], rtol=0, atol=0), "routed weights placed"
    assert np.allclose(g["wts"][-x.shape[0]:], r["gamma"], rtol=0, atol=1e-6), "shared gate"


def test_prefill_timed_matches_prefill(moe):
    """moe_prefill_timed runs the same kernels as moe_prefill (the same ids;
    the same bf16 output up to one ulp, since the down GEMM's scatter adds in
    fp32 in whatever order its tiles finish) and records its events around
    each of them, in order: the per-kernel times add up to the whole call."""
    rng = np.random.default_rng(880)
    H, E, k, I, t = 512, 16, 4, 256, 300
    layer = synth.make_layer(rng, H, E, k, I, 4, shared=True, flags=synth.RESIDUAL)
    dl = moe.DeviceLayers([layer])
    x = rng.normal(size=(t, H)).astype(np.float32)
    o_ref, idx_ref = run_prefill(moe, dl, x)
    xt = torch.from_numpy(x).cuda()
    out = torch.empty((t, H), dtype=torch.int16, device="cuda")
    idx = torch.zeros((t, k), dtype=torch.int32, device="cuda")
    ws = moe.alloc_workspace(moe.prefill_workspace(dl, t))
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    stream = torch.cuda.current_stream()
    evs = [torch.cuda.Event(enable_timing=True) for _ in range(moe.PREFILL_KERNELS + 1)]
    for e in evs:
        e.record(stream)
    torch.cuda.synchronize()
    moe.prefill_timed(dl, xt, out, ws, status, evs, idx, stream=stream)
    torch.cuda.synchronize()
    assert status.item() == 0, moe.STATUS_NAMES.get(status.item())
    o = synth.bf16_bits_to_f32(out.cpu().numpy().view(np.uint16)).astype(np.float64)
    assert np.array_equal(idx.cpu().numpy(), idx_ref)
    assert (np.abs(o - o_ref) <= bf16_ulp(o_ref)).all()
    parts = [evs[j].elapsed_time(evs[j + 1]) for j in range(moe.PREFILL_KERNELS)]
    total = evs[0].elapsed_time(evs[-1])
    assert all(p >= 0 for p in parts) and abs(sum(parts) - total) <= 1e-3 * max(total, 1.0)
    print(f"[prefill] timed call: {moe.PREFILL_KERNELS} kernels, {total * 1e3:.1f} us, outputs equal the plain call")


def test_prefill_zero_rows_route_by_the_tie_rule(moe):
    """Rows of zeros in a chunk: every logit is 0, so the k experts are the k
    lowest ids (ties go to the lower id) and the row's output is exactly
    zero; the other rows still match the oracle."""
    rng = np.random.default_rng(1210)
    H, E, k, I, t = 256, 16, 4, 128, 40
    layer = synth.make_layer(rng, H, E, k, I, 4, shared=True, flags=synth.RESIDUAL | synth.PRENORM)
    ol = oracle.Layer(layer)
    x = rows_with_gap(ol, rng, t, H)
    zero = np.arange(0, t, 3)
    x[zero] = 0.0
    got, idx = run_prefill(moe, moe.DeviceLayers([layer]), x)
    assert (idx[zero] == np.arange(k)).all(), idx[zero]
    assert np.all(got[zero] == 0.0)
    rest = np.setdiff1d(np.arange(t), zero)
    ref = oracle.prefill_rows(ol, x, rest, mirror=True)
    assert np.array_equal(np.sort(idx[rest], axis=1), np.sort(ref["idx"], axis=1))
    assert_prefill_close(got[rest], ref, x, layer.flags, rest, "rows beside zero rows")
