"""The no-allocation per-tensor FP8 entry point, called through the C ABI.

Some callers of this library cannot allocate device memory or pass a
workspace (a plugin inside a serving engine whose device memory is already
reserved for the engine's own pool, or code that must keep its memory
footprint fixed after start-up).  qlin_quantize_fp8_tensor_noalloc keeps its
scratch in a fixed device array inside the library; these tests check that
it produces exactly what the workspace-based entry point produces, on two
calls in a row (the second call sees the first call's leftovers in the shared
array), and that it refuses tensors larger than that array can serve.
"""
import numpy as np
import pytest
import torch

from gpu_util import require_gpu
from serving_amax_reduce_gb300 import inputs

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def q():
    return require_gpu()


def noalloc(q, x):
    M, K = x.shape
    codes = torch.empty(M * K, dtype=torch.uint8, device=x.device)
    scale = torch.empty(1, dtype=torch.float32, device=x.device)
    rc = q.qlin_quantize_fp8_tensor_noalloc(x.data_ptr(), M, K, x.stride(0), codes.data_ptr(), scale.data_ptr(),
                                            torch.cuda.current_stream().cuda_stream)
    assert rc == 0, q.qlin_status_string(rc)
    return codes, scale


def test_noalloc_matches_workspace_entry_point_on_two_calls(q):
    # first call: a large-amax tensor; second: smaller tensor, smaller amax, so
    # any stale partial left in the shared array would change its scale
    cases = [inputs.normal_bf16((4096, 4096), 3.0, 71), inputs.normal_bf16((128, 1024), 0.02, 72)]
    for x in cases:
        xd = x.cuda()
        ref = q.quantize_act(q.Fmt.FP8_TENSOR, xd)
        codes, scale = noalloc(q, xd)
        torch.cuda.synchronize()
        assert torch.equal(codes, ref["codes"][: codes.numel()])
        assert scale.view(torch.int32).item() == ref["scales"][:1].view(torch.int32).item()


def test_noalloc_at_its_largest_size(q):
    """rows * K equal to the limit: every slot of the fixed array, the last
    one included, is written and read; the result equals the workspace entry
    point's bit for bit.  One row more at the same K is refused."""
    K = 4096
    rows = q.NOALLOC_MAX_ELEMENTS // K
    x = inputs.normal_bf16((rows, K), 1.0, 73)
    x[-1, -1] = 40.0                         # the tensor amax sits in the last partial's block
    xd = x.cuda()
    ref = q.quantize_act(q.Fmt.FP8_TENSOR, xd)
    codes, scale = noalloc(q, xd)
    torch.cuda.synchronize()
    assert torch.equal(codes, ref["codes"][: codes.numel()])
    assert scale.view(torch.int32).item() == ref["scales"][:1].view(torch.int32).item()
    assert scale.view(torch.int32).item() == int(np.array([np.float32(40) / np.float32(448)]).view(np.int32)[0])
    st = torch.cuda.current_stream().cuda_stream
    assert q.qlin_quantize_fp8_tensor_noalloc(xd.data_ptr(), rows + 1, K, K, codes.data_ptr(), scale.data_ptr(),
                                              st) == q.Status.WORKSPACE


def test_noalloc_rejects_tensors_beyond_its_scratch(q):
    S = q.Status
    x = torch.zeros(16, dtype=torch.bfloat16, device="cuda")
    st = torch.cuda.current_stream().cuda_stream
    rows = q.NOALLOC_MAX_ELEMENTS // 1024 + 1
    # rejected on the host before any launch: the pointers are never touched
    assert q.qlin_quantize_fp8_tensor_noalloc(x.data_ptr(), rows, 1024, 1024, x.data_ptr(), x.data_ptr(),
                                              st) == S.WORKSPACE
    assert q.qlin_quantize_fp8_tensor_noalloc(None, 8, 1024, 1024, x.data_ptr(), x.data_ptr(), st) == S.INVALID_ARG
