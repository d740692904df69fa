"""The allocation-free projection forward (lr_proj_fwd_noalloc).

Some callers cannot call cudaMalloc (a framework allocator owns device memory,
a memory budget forbids new allocations, or the code must not synchronise the
device), so they cannot hand lr_proj_fwd a workspace.  lr_proj_fwd_noalloc
keeps its scratch in a fixed device array inside the library.  This test calls
it through the C ABI twice in a row, with different shapes, and checks each
result against lr_proj_fwd on the same inputs.  Both entry points launch the
same kernels on the same inputs (only the place of the folded weights
differs), so the outputs and the saved set must agree bit for bit.  It lives in
a file collected last so that a run stopping at the first failure has already
run every other test.
"""
import pytest
import torch

from rank_bottleneck_block_gb300 import inputs as I

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    from rank_bottleneck_block_gb300 import build

    build.build()


def test_proj_fwd_noalloc_matches_proj_fwd_twice():
    from rank_bottleneck_block_gb300 import lowrank as L
    from rank_bottleneck_block_gb300.runner import ProjGroup

    shapes = [
        I.ProjShape(T=1000, d_in=1024, d_out=768, r=256, group=3, norm=True),
        I.ProjShape(T=300, d_in=520, d_out=264, r=72, group=1, norm=False),
    ]
    for call, shape in enumerate(shapes):
        case = I.make_proj_case(shape, seed=11 + call, with_grad=False)
        ref = ProjGroup(shape, case)
        ref.saved.zero_()  # the saved set's alignment padding is never written: start both at zero
        ref.forward()
        outs = [torch.empty_like(o) for o in ref.outs]
        saved = torch.zeros_like(ref.saved)
        L.lr_proj_fwd_noalloc(ref.dt, shape.T, shape.d_in, shape.d_out, shape.r, ref.pairs(), ref.g, shape.eps,
                              ref.x, outs, saved)
        torch.cuda.synchronize()
        L.lr_check_device_error()
        for i in range(shape.group):
            assert torch.equal(outs[i], ref.outs[i]), (call, i)
        assert torch.equal(saved, ref.saved), call


def test_proj_fwd_noalloc_rejects_oversized_scratch():
    from rank_bottleneck_block_gb300 import lowrank as L

    # 3 * 2048 * 4096 bf16 weights = 48 MiB > the 32 MiB array: rejected before any launch
    T, d_in, d_out, r, group = 64, 4096, 64, 2048, 3
    p = torch.empty(16, dtype=torch.bfloat16, device="cuda")
    saved = torch.empty(L.lr_proj_saved_bytes(L.LR_BF16, T, d_in, d_out, r, group, 0), dtype=torch.uint8,
                        device="cuda")
    with pytest.raises(L.LowRankError) as ei:
        L.lr_proj_fwd_noalloc(L.LR_BF16, T, d_in, d_out, r, [L.pair(p, p)] * group, None, 1e-6, p, [p] * group,
                              saved)
    assert ei.value.status == 5 and "scratch" in str(ei.value)
