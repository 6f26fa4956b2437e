"""dsv4_o_proj_static: the O-projection for callers that cannot allocate device
memory (an engine plugin handed no allocator, or a latency path where
cudaMalloc would synchronise the device).  It must give the same output as
dsv4_o_proj with a caller workspace, call after call, and reject sizes beyond
its fixed scratch.  This file is collected last on purpose."""
import pytest
import torch

import dsv4_inputs as di
from gpu_helpers import GEMM_RTOL, cuda_or_skip, gemm_rel_err, to_bits

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def dev():
    return cuda_or_skip()


def _static_call(lib, d, w, out):
    return lib.dsv4_o_proj_static(
        d["o"].data_ptr(), d["positions"].data_ptr(), d["cache"].data_ptr(), w.max_pos, w.T,
        w.n_groups, w.heads_per_group, 448, 64, 128, w.o_lora_rank, w.hidden,
        d["wo_a"].data_ptr(), d["wo_a_scale"].data_ptr(), d["wo_b"].data_ptr(),
        d["wo_b_scale"].data_ptr(), out.data_ptr(), torch.cuda.current_stream().cuda_stream)


@pytest.mark.parametrize("name,T", [("full", 256), ("full", 77), ("tiny", 16)])
def test_static_matches_workspace_entry_twice(dev, name, T):
    import deepseek_v4_attention_gb300 as k
    lib = k.load_library()
    w = di.WORKLOADS[name].with_tokens(T, seed=T + 5)
    d = {n: t.to(dev) for n, t in di.make_inputs(w).items()}
    ref = k.dsv4_o_proj(d["o"], d["positions"], d["cache"], d["wo_a"], d["wo_a_scale"],
                        d["wo_b"], d["wo_b_scale"], n_groups=w.n_groups,
                        heads_per_group=w.heads_per_group, o_lora_rank=w.o_lora_rank)
    torch.cuda.synchronize()
    ref_bits = to_bits(ref)
    ref64 = ref.double().cpu().numpy()
    for _ in range(2):                     # two calls in a row share the same scratch
        out = torch.full((w.T, w.hidden), float("nan"), dtype=torch.bfloat16, device=dev)
        assert _static_call(lib, d, w, out) == 0
        assert k.dsv4_last_launch_count() == 3
        torch.cuda.synchronize()
        assert k.dsv4_device_status(clear=True) == 0
        bits = to_bits(out)
        assert gemm_rel_err(bits, ref64) <= GEMM_RTOL
        assert (bits == ref_bits).all()    # same kernels, same order: identical


def test_static_rejects_sizes_beyond_its_scratch(dev):
    import deepseek_v4_attention_gb300 as k
    lib = k.load_library()
    w = di.WORKLOADS["full"].with_tokens(813)       # 82.5 KB/token: one token too many
    assert k.dsv4_o_proj_workspace_bytes(813, 16, 8, 512, 1024) > k.static_scratch_bytes()
    assert k.dsv4_o_proj_workspace_bytes(812, 16, 8, 512, 1024) <= k.static_scratch_bytes()
    d = {n: t.to(dev) for n, t in di.make_inputs(w).items()}
    out = torch.zeros((w.T, w.hidden), dtype=torch.bfloat16, device=dev)
    assert _static_call(lib, d, w, out) == k._NAME_TO_CODE["DSV4_ERR_WORKSPACE"]
    assert k.dsv4_last_launch_count() == 0
    torch.cuda.synchronize()
    assert bool((out == 0).all())          # nothing was written


def test_static_calls_allocate_nothing(dev):
    """After a first call (which looks up the scratch's device address), further
    calls change neither the device's free memory nor torch's allocations."""
    import deepseek_v4_attention_gb300 as k
    lib = k.load_library()
    w = di.WORKLOADS["full"].with_tokens(128, seed=9)
    d = {n: t.to(dev) for n, t in di.make_inputs(w).items()}
    out = torch.empty((w.T, w.hidden), dtype=torch.bfloat16, device=dev)
    assert _static_call(lib, d, w, out) == 0
    torch.cuda.synchronize()
    free0, _ = torch.cuda.mem_get_info(dev)
    alloc0 = torch.cuda.memory_allocated(dev)
    for _ in range(5):
        assert _static_call(lib, d, w, out) == 0
    torch.cuda.synchronize()
    assert k.dsv4_device_status(clear=True) == 0
    assert torch.cuda.mem_get_info(dev)[0] == free0
    assert torch.cuda.memory_allocated(dev) == alloc0
