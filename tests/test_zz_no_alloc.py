"""kascade_dense_decode_noalloc: dense decode for callers that cannot allocate.

Some callers cannot call cudaMalloc (their device memory belongs to another
allocator, or they run where allocation is not allowed), so they cannot hand
the library a workspace. This entry point keeps its scratch in a fixed
device array inside the library instead. The test calls it through the C ABI
twice in a row, on different inputs, and checks each result against the
float64 oracle within the decode tolerances, and for equality, bit for bit,
with the workspace-based kascade_dense_decode (the same kernel with the same
split count). The array's error word, read through
kascade_noalloc_device_error, must stay clear. The file sits on its own and
is collected last; it passes alone or after the other tests.
"""
import ctypes

import pytest
import torch

import __graft_entry__
from gpu_helpers import check_out, f64
from oracle import attention as A

pytestmark = pytest.mark.gpu


def _layer(seed, B, Hq, Hkv, N, d):
    g = torch.Generator().manual_seed(seed)
    q = torch.randn(B, Hq, d, generator=g)
    k = torch.randn(B, Hkv, N, d, generator=g)
    v = torch.randn(B, Hkv, N, d, generator=g)
    return [x.to(torch.bfloat16).cuda() for x in (q, k, v)]


@pytest.mark.parametrize("shape", [(2, 8, 2, 3000, 128), (1, 16, 2, 5000, 64)])
def test_noalloc_matches_oracle_on_two_calls(shape):
    __graft_entry__.build()
    from long_context_anchor_gb300 import kascade as K
    fn = K._lib.kascade_dense_decode_noalloc
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    for call, seed in enumerate((11, 12)):
        q, k, v = _layer(seed + shape[3], *shape)
        out = torch.full_like(q, float("nan"))
        desc = K.decode_desc(q, k)
        st = fn(ctypes.byref(desc), ctypes.c_void_p(q.data_ptr()), ctypes.c_void_p(k.data_ptr()),
                ctypes.c_void_p(v.data_ptr()), ctypes.c_void_p(out.data_ptr()), stream)
        assert st == K.OK, (call, K.status_string(st))
        assert K._lib.kascade_noalloc_device_error(stream) == K.OK, call
        o_ref, _ = A.dense_decode(f64(q), f64(k), f64(v))
        check_out(out, o_ref, what=("noalloc", call))
        assert torch.equal(out, K.dense_decode(q, k, v)), call
