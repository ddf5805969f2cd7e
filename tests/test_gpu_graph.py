"""Device-buffer calls captured in a CUDA graph replay to the same bits as eager calls.

A launch-bound sequence of small GEMMs is the case for graphs: the host cost of each
call (argument checks, tensor-map cache lookups, launch) is paid once at capture.  The
handle is bound, and any workspace grown, by an eager call of the same shapes before
capture (the calls themselves make no allocation then).
"""
import pytest
import torch

import mixed_precision_tensor_gb300 as tcg

pytestmark = pytest.mark.gpu

N, T = tcg.TCG_OP_N, tcg.TCG_OP_T

CASES = [
    # m, n, k, in, compute, out: a plain tile grid, a split-K shape, TF32 and the
    # three-product TF32 split (both round into the workspace first)
    (512, 768, 320, torch.float16, tcg.TCG_COMPUTE_32F, torch.float32),
    (256, 256, 16384, torch.bfloat16, tcg.TCG_COMPUTE_32F, torch.bfloat16),
    (384, 640, 1000, torch.float32, tcg.TCG_COMPUTE_32F_FAST_TF32, torch.float32),
    (384, 640, 1000, torch.float32, tcg.TCG_COMPUTE_32F_3XTF32, torch.float32),
]


def _code(dt):
    return {torch.float16: tcg.TCG_R_16F, torch.bfloat16: tcg.TCG_R_16BF,
            torch.float32: tcg.TCG_R_32F}[dt]


# (case, TF32 rounding mode): every case with the default rounding, and the TF32 case also
# through the in-kernel rounding option, whose counters a memset node zeroes before each
# GEMM launch
GRAPH_CASES = [c + (0,) for c in CASES] + [CASES[2] + (2,)]


@pytest.mark.parametrize("m,n,k,in_dt,compute,out_dt,tf32_rounding", GRAPH_CASES)
def test_graph_replay_matches_eager(cuda_device, m, n, k, in_dt, compute, out_dt, tf32_rounding):
    gen = torch.Generator(device="cpu").manual_seed(m + n + k)
    A = (torch.rand(k, m, generator=gen) * 2 - 1).to(in_dt).cuda()       # column-major m x k
    B = (torch.rand(n, k, generator=gen) * 2 - 1).to(in_dt).cuda()       # column-major k x n
    C0 = (torch.rand(n, m, generator=gen) * 2 - 1).to(out_dt).cuda()     # column-major m x n
    stream = torch.cuda.Stream()
    h = tcg.Handle(stream)
    tcg.check(tcg.tcg_set_tf32_rounding(h.h, tf32_rounding))

    def chain(C):
        # three dependent calls: D = A B + 0.5 D, D is C
        for _ in range(3):
            tcg.check(tcg.tcg_gemm_ex(h.h, N, N, m, n, k, 1.0, A, _code(in_dt), m, B,
                                      _code(in_dt), k, 0.5, C, _code(out_dt), m, compute))

    eager = C0.clone()
    with torch.cuda.stream(stream):
        chain(eager)                       # binds the handle and grows its workspace
    stream.synchronize()
    tcg.check(tcg.tcg_get_device_error(h.h))

    Cg = C0.clone()
    graph = torch.cuda.CUDAGraph()
    launches_before = tcg.tcg_launch_count(h.h)
    with torch.cuda.graph(graph, stream=stream):
        chain(Cg)
    captured = tcg.tcg_launch_count(h.h) - launches_before
    assert captured >= 3
    torch.cuda.synchronize()
    Cg.copy_(C0)                           # capture ran nothing: start from C0
    for _ in range(2):                     # replays are repeatable
        Cg.copy_(C0)
        graph.replay()
        torch.cuda.synchronize()
        tcg.check(tcg.tcg_get_device_error(h.h))
        assert torch.equal(Cg.view(torch.uint8) if out_dt != torch.float32 else Cg.view(torch.int32),
                           eager.view(torch.uint8) if out_dt != torch.float32 else eager.view(torch.int32))
    h.close()
