"""bsp_attention_host: attention on host tensors with the batch cut into
slices whose copies overlap the kernels.  The output must equal bsp_attention
on the same data copied to the device (identical bytes: the same kernels run
on each slice), for several batch sizes, slice sizes, pinned and pageable
host memory, both tensor-core and CUDA-core paths; and a small case against
the fp64 oracle."""

import numpy as np
import pytest
import torch

from gpu_util import TOL, normwise_err, to_np
from sparse_attention_layout_gb300 import workloads as W

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def bsp():
    if not torch.cuda.is_available():
        pytest.skip("no GPU")
    from sparse_attention_layout_gb300 import build
    build.build()
    from sparse_attention_layout_gb300 import bsp as m
    return m


@pytest.mark.parametrize("Z,z_slice", [(1, 1), (3, 1), (4, 1), (5, 2), (4, 4)])
@pytest.mark.parametrize("pinned", [True, False])
@pytest.mark.parametrize("dt", ["bf16", "f32"])
def test_host_equals_device(bsp, Z, z_slice, pinned, dt):
    B, nb, H, D = 64, 6, 3, 64
    lay = W.layout_strided_causal(nb, 2, 3, H)
    L = bsp.bsp_layout_compile(lay, B)
    S = nb * B
    Q, K, V = (W.randn((Z, H, S, D), dt, 400 + s) for s in range(3))
    if pinned:
        Q, K, V = (t.pin_memory() for t in (Q, K, V))
    O = torch.empty_like(Q).pin_memory() if pinned else torch.empty_like(Q)
    ws = torch.empty(bsp.bsp_attention_host_workspace(L, Q.dtype, D, z_slice), dtype=torch.uint8, device="cuda")
    bsp.bsp_attention_host(L, Q, K, V, O, 0.125, W.MASK_DIAG_CAUSAL, workspace=ws)
    torch.cuda.synchronize()
    want = bsp.bsp_attention(L, Q.cuda(), K.cuda(), V.cuda(), None, 0.125, W.MASK_DIAG_CAUSAL)
    torch.cuda.synchronize()
    assert torch.equal(O, want.cpu())


def test_host_against_oracle_and_mask(bsp, oracle):
    B, nb, H, D, Z = 32, 8, 2, 128, 3
    lay = (np.random.default_rng(5).random((H, nb, nb)) < 0.4).astype(np.uint8)
    L = bsp.bsp_layout_compile(lay, B)
    S = nb * B
    Q, K, V = (W.randn((Z, H, S, D), "f16", 410 + s).pin_memory() for s in range(3))
    mask = W.random_mask(S, 0.7, 413)
    O = bsp.bsp_attention_host(L, Q, K, V, None, 0.09, W.MASK_DENSE, torch.from_numpy(mask).cuda())
    torch.cuda.synchronize()
    want = oracle.attention(lay, B, Q, K, V, 0.09, W.MASK_DENSE, mask)
    assert normwise_err(to_np(O), want) <= TOL[torch.float16]


def test_host_rejects_small_workspace_and_device_tensors(bsp):
    lay = np.ones((1, 4, 4), np.uint8)
    L = bsp.bsp_layout_compile(lay, 32)
    Q = torch.randn(2, 1, 128, 64, dtype=torch.bfloat16)
    small = torch.empty(bsp.bsp_attention_host_workspace(L, Q.dtype, 64, 1) - 256, dtype=torch.uint8, device="cuda")
    with pytest.raises(bsp.BspError) as e:
        bsp.bsp_attention_host(L, Q, Q, Q, None, 0.1, workspace=small)
    assert e.value.code == -1
    with pytest.raises(ValueError):
        bsp.bsp_attention_host(L, Q.cuda(), Q, Q)


@pytest.mark.parametrize("reserved", [False, True])
def test_host_repeated_calls_reuse_slots(bsp, reserved):
    # several calls in a row on one handle (the slot hand-off events are reused;
    # with a reserved workspace a call's input copies overlap the previous
    # call's tail)
    B, nb, H, D, Z = 128, 4, 2, 64, 6
    L = bsp.bsp_layout_compile(W.layout_band(nb, 1, H), B)
    S = nb * B
    ws = torch.empty(bsp.bsp_attention_host_workspace(L, torch.bfloat16, D, 1), dtype=torch.uint8, device="cuda")
    outs = []
    for rep in range(4):
        Q, K, V = (W.randn((Z, H, S, D), "bf16", 420 + 3 * rep + s).pin_memory() for s in range(3))
        O = bsp.bsp_attention_host(L, Q, K, V, None, 0.125, workspace=ws, reserved_workspace=reserved)
        outs.append((O, Q, K, V))
    torch.cuda.synchronize()
    for O, Q, K, V in outs:
        assert torch.equal(O, bsp.bsp_attention(L, Q.cuda(), K.cuda(), V.cuda(), None, 0.125).cpu())


def test_host_reserved_workspace_calls_of_changing_slot_size(bsp):
    # calls on one handle and one reserved workspace whose slots change size
    # from call to call (batch size, so the slicing, and head size change): a
    # call whose slots differ from the previous call's must not start its
    # input copies before that call's kernels and output copies are done, since
    # its slot 0 can cover the previous call's slot 1
    B, nb, H = 64, 4, 2
    L = bsp.bsp_layout_compile(W.layout_band(nb, 1, H), B)
    S = nb * B
    ws = torch.empty(bsp.bsp_attention_host_workspace(L, torch.bfloat16, 128, 2), dtype=torch.uint8,
                     device="cuda")
    outs = []
    for rep, (Z, D) in enumerate([(4, 128), (6, 64), (2, 64), (5, 128), (8, 64), (3, 128), (4, 128)]):
        Q, K, V = (W.randn((Z, H, S, D), "bf16", 430 + 3 * rep + s).pin_memory() for s in range(3))
        O = bsp.bsp_attention_host(L, Q, K, V, None, 0.125, workspace=ws, reserved_workspace=True)
        outs.append((O, Q, K, V))
    torch.cuda.synchronize()
    for O, Q, K, V in outs:
        assert torch.equal(O, bsp.bsp_attention(L, Q.cuda(), K.cuda(), V.cuda(), None, 0.125).cpu())
