"""The allocation-free entry point (moe_forward_noalloc) against moe_forward.

Some callers cannot allocate device memory while they run the step (graph
capture, engines that own all device memory, loops that must not risk an
allocation's implicit synchronisation); moe_forward_noalloc serves them from
a fixed array inside the library.  This file is collected last on purpose."""
import numpy as np
import pytest

from helpers import TOL, assert_close_rows
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


def test_noalloc_matches_workspace_call_twice(moe):
    layers = synth.make_config_layers("c1", seed=7, n_layers=4)
    dl = moe.DeviceLayers(layers)
    nb, H, k = 2, 2048, 8
    x = torch.from_numpy(synth.make_x(np.random.default_rng(8), nb, H, rho=0.3)).cuda()
    status = torch.zeros(1, dtype=torch.int32, device="cuda")

    ref = torch.empty_like(x)
    ws = moe.alloc_workspace(moe.forward_workspace(dl, nb))
    slot_r = torch.zeros((4, 64), dtype=torch.int64, device="cuda")
    idx_r = torch.zeros((4, nb, k), dtype=torch.int32, device="cuda")
    moe.forward(dl, x, ref, ws, status, slot_r, None, idx_r)
    torch.cuda.synchronize()
    assert status.item() == 0
    ref_np = ref.cpu().numpy().astype(np.float64)
    layer_moe = ref_np - x.cpu().numpy()  # stream growth over 4 layers sets the scale

    for call in range(2):
        out = torch.full_like(x, float("nan"))
        slot = torch.zeros((4, 64), dtype=torch.int64, device="cuda")
        idx = torch.zeros((4, nb, k), dtype=torch.int32, device="cuda")
        moe.forward_noalloc(dl, x, out, status, slot, None, idx)
        torch.cuda.synchronize()
        assert status.item() == 0, f"call {call}"
        assert torch.equal(idx, idx_r), f"call {call}: routed ids"
        assert torch.equal(slot, slot_r), f"call {call}: slot table"
        assert_close_rows(out.cpu().numpy(), ref_np, layer_moe, tol=TOL, what=f"noalloc call {call}")


def test_noalloc_rejects_layers_beyond_its_scratch(moe):
    # 64 layers of hidden 2048 / 512 experts need more than the fixed scratch
    # at nb 4.  One small layer (inter 128) is uploaded once and its ABI struct
    # repeated 64 times: the size check runs on the host before anything reads
    # the weights.
    L = synth.make_layer(np.random.default_rng(0), 2048, 512, 10, 128, 4, shared=True)
    one = moe.DeviceLayers([L])

    class Stack:
        c = (moe.MoeLayer * 64)(*([one.c[0]] * 64))
        n = 64

    need = moe.forward_workspace(Stack.c, 4)
    assert need > moe.NOALLOC_MAX_WORKSPACE
    x = torch.zeros((4, 2048), device="cuda")
    out = torch.empty_like(x)
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    with pytest.raises(moe.MoeError) as e:
        moe.forward_noalloc(Stack, x, out, status)
    assert e.value.code == moe.ENOSPACE
