"""The number of kernels a forward call enqueues equals what the library
plans (awq_forward_launches), counted from the CUDA kernel records of the
PyTorch profiler; the stream-K sum kernel runs exactly when a tile of the
last partial wave is split along k, which the prefill path does unless that
wave already fills most SMs (then its tiles run whole, one per CTA)."""
import pytest
import torch

import bit_weight_quantized_awq_gb300 as awq
from bit_weight_quantized_awq_gb300 import Path
from bit_weight_quantized_awq_gb300.synthetic import make_problem

pytestmark = pytest.mark.gpu

CASES = [
    # (M, K, N, g, path, split): split = the sum kernel runs (on 152 SMs)
    (1, 4096, 4096, 128, Path.AUTO, False),          # decode
    (64, 8192, 10240, 128, Path.AUTO, True),         # fused prefill, every tile split
    (512, 4096, 12288, 128, Path.PREFILL, True),     # 96 tiles, split
    (128, 4096, 38912, 128, Path.PREFILL, False),    # 152 whole tiles: no last wave
    (2048, 4096, 12288, 128, Path.AUTO, True),       # 2 waves + 80 split tiles
    (2048, 4096, 4096, 128, Path.AUTO, False),       # 128 tiles: the wave runs whole
    (512, 8192, 57344, 128, Path.PREFILL, False),    # 2 waves + 144 tiles run whole
    (8192, 4096, 12288, 128, Path.AUTO, True),       # dequant + GEMM
    (2048, 11008, 4096, 128, Path.DEQUANT_GEMM, True),
]


@pytest.fixture(scope="module", autouse=True)
def profiler_warm():
    # the first profiler session of a process may miss kernels while the
    # tracing library starts up: run one on a plain torch op first
    acts = [torch.profiler.ProfilerActivity.CPU, torch.profiler.ProfilerActivity.CUDA]
    with torch.profiler.profile(activities=acts):
        torch.ones(1024, device="cuda").sum()
        torch.cuda.synchronize()


def awq_kernels(prof):
    names = [e.name for e in prof.events()
             if e.device_type == torch.autograd.DeviceType.CUDA and "awq" in e.name]
    return names


@pytest.mark.parametrize("M,K,N,g,path,split", CASES)
def test_kernels_per_call_match_the_plan(M, K, N, g, path, split):
    dev = torch.device("cuda")
    p = make_problem(M, K, N, g, bias=False, seed=0).to(dev)
    y = torch.empty((M, N), dtype=torch.float16, device=dev)
    awq.linear_forward(p.x, p.qweight, p.qzeros, p.scales, None, g, path=path, out=y)
    torch.cuda.synchronize()
    acts = [torch.profiler.ProfilerActivity.CPU, torch.profiler.ProfilerActivity.CUDA]
    with torch.profiler.profile(activities=acts) as prof:
        awq.linear_forward(p.x, p.qweight, p.qzeros, p.scales, None, g, path=path, out=y)
        torch.cuda.synchronize()
    names = awq_kernels(prof)
    if not names:
        pytest.skip("the profiler recorded no CUDA kernels here")
    want = awq.awq_forward_launches(M, K, N, g, path)
    assert len(names) == want, names
    n_sum = sum("sk_fixup_kernel" in n for n in names)
    used = Path(awq.awq_select_path(M, K, N, g)) if path == Path.AUTO else path
    if used == Path.PREFILL:
        assert n_sum == want - 1
    elif used != Path.DEQUANT_GEMM:
        assert n_sum == 0
    if torch.cuda.get_device_properties(dev).multi_processor_count == 152:
        assert (n_sum > 0) == split, names
