"""kascade_dense_decode_noalloc: dense decode for callers that cannot allocate.

Some callers cannot call cudaMalloc (their device memory belongs to another
allocator, or they run where allocation is not allowed), so they cannot hand
the library a workspace. This entry point keeps its scratch in a fixed
device array inside the library instead. The test calls it through the C ABI
twice in a row, on different inputs, and checks each result against the
workspace-based kascade_dense_decode within the decode tolerances. It sits
in a file of its own, collected last, and passes alone or after the others.
"""
import ctypes

import pytest
import torch

import __graft_entry__

pytestmark = pytest.mark.gpu

MAX_ABS, MEAN_ABS = 2e-2, 2e-3


def _layer(seed, B, Hq, Hkv, N, d):
    g = torch.Generator().manual_seed(seed)
    q = torch.randn(B, Hq, d, generator=g)
    k = torch.randn(B, Hkv, N, d, generator=g)
    v = torch.randn(B, Hkv, N, d, generator=g)
    return [x.to(torch.bfloat16).cuda() for x in (q, k, v)]


@pytest.mark.parametrize("shape", [(2, 8, 2, 3000, 128), (1, 16, 2, 5000, 64)])
def test_noalloc_matches_dense_decode_on_two_calls(shape):
    __graft_entry__.build()
    from long_context_anchor_gb300 import kascade as K
    fn = K._lib.kascade_dense_decode_noalloc
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    for call, seed in enumerate((11, 12)):
        q, k, v = _layer(seed + shape[3], *shape)
        ref = K.dense_decode(q, k, v)
        out = torch.full_like(q, float("nan"))
        desc = K.decode_desc(q, k)
        st = fn(ctypes.byref(desc), ctypes.c_void_p(q.data_ptr()), ctypes.c_void_p(k.data_ptr()),
                ctypes.c_void_p(v.data_ptr()), ctypes.c_void_p(out.data_ptr()), stream)
        assert st == K.OK, (call, K.status_string(st))
        torch.cuda.synchronize()
        err = (out.float() - ref.float()).abs()
        assert torch.isfinite(out.float()).all(), call
        assert err.max().item() <= MAX_ABS and err.mean().item() <= MEAN_ABS, (call, err.max().item())
