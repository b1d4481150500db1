"""dflash2_unary_topk_noalloc against dflash2_unary_topk, through the C-ABI.

The no-allocation entry point serves callers that may not allocate device memory
during a call (a host framework that owns all device memory, a latency-critical
path where cudaMalloc's possible device synchronisation is not acceptable).  It
must give the same top-K ids, values and G as the workspace entry point, on two
calls in a row: the second call finds the first call's leftovers in the shared
scratch array.  This file is collected last on purpose."""
import ctypes as ct

import numpy as np
import pytest

from parity import close

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu


def _p(t):
    return ct.c_void_p(0 if t is None else t.data_ptr())


@pytest.fixture(scope="module")
def lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from dflash2_draft_block_gb300 import _abi, build
    build.build()
    return _abi.load()


def _inputs(seed, P, D, V, r):
    g = torch.Generator().manual_seed(seed)
    h = torch.randn((P, D), generator=g).to(torch.bfloat16).cuda()
    W = (torch.randn((V, D), generator=g) * 0.02).to(torch.bfloat16).cuda()
    WH = (torch.randn((r, D), generator=g) * 0.02).to(torch.bfloat16).cuda()
    return h, W, WH


def _with_workspace(lib, h, W, K, WH, stream):
    P, D = h.shape
    V, r = W.shape[0], WH.shape[0]
    ids = torch.empty((P, K), dtype=torch.int32, device="cuda")
    vals = torch.empty((P, K), dtype=torch.float32, device="cuda")
    G = torch.empty((P, r), dtype=torch.float32, device="cuda")
    nbytes = lib.dflash2_unary_topk_workspace_size(P, D, V, K, r)
    ws = torch.empty(max(nbytes, 1), dtype=torch.uint8, device="cuda")
    rc = lib.dflash2_unary_topk(_p(h), P, D, _p(W), V, K, 1.0, 0.0, _p(WH), r, _p(G), _p(ids), _p(vals), _p(ws),
                                nbytes, None, stream)
    assert rc == 0, lib.dflash2_status_string(rc)
    return ids, vals, G


def _no_alloc(lib, h, W, K, WH, stream):
    P, D = h.shape
    V, r = W.shape[0], WH.shape[0]
    ids = torch.full((P, K), -7, dtype=torch.int32, device="cuda")
    vals = torch.zeros((P, K), dtype=torch.float32, device="cuda")
    G = torch.zeros((P, r), dtype=torch.float32, device="cuda")
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    rc = lib.dflash2_unary_topk_noalloc(_p(h), P, D, _p(W), V, K, 1.0, 0.0, _p(WH), r, _p(G), _p(ids), _p(vals),
                                        _p(status), stream)
    assert rc == 0, lib.dflash2_status_string(rc)
    return ids, vals, G, status


STREAM, GEMM, CUDA_CORE = 0, 1, 2   # DF2_HEAD_PATH_*


@pytest.mark.parametrize("shape", [
    # (P, D, V, K, r, head path)
    [(8, 4096, 151936, 16, 256, STREAM), (8, 4096, 151936, 16, 256, STREAM)],   # batch-1 head, twice
    [(8, 512, 30011, 16, 64, STREAM), (24, 256, 5000, 64, 32, GEMM)],           # different shapes back to back
    [(40, 256, 3000, 8, 32, GEMM), (5, 1024, 7777, 32, 128, STREAM)],           # GEMM path, then streaming
    [(20, 256, 3000, 100, 32, CUDA_CORE), (9, 512, 20011, 64, 64, STREAM)],     # CUDA-core path (K > 64)
    # the GEMM path keeps a per-position threshold in the scratch: a larger call,
    # then a smaller one that must not see the first call's thresholds
    [(256, 512, 40000, 16, 64, GEMM), (64, 512, 9000, 16, 64, GEMM)],
])
def test_no_alloc_matches_workspace_entry_point(lib, shape):
    stream = ct.c_void_p(torch.cuda.current_stream().cuda_stream)
    for i, (P, D, V, K, r, path) in enumerate(shape):
        assert lib.dflash2_unary_topk_path(P, D, V, K) == path
        h, W, WH = _inputs(100 * i + P, P, D, V, r)
        ref_ids, ref_vals, ref_G = _with_workspace(lib, h, W, K, WH, stream)
        ids, vals, G, status = _no_alloc(lib, h, W, K, WH, stream)
        torch.cuda.synchronize()
        assert int(status.item()) == 0
        assert torch.equal(ids, ref_ids)
        close(vals.cpu().numpy(), ref_vals.cpu().numpy(), what="no-alloc vals")
        close(G.cpu().numpy(), ref_G.cpu().numpy(), what="no-alloc G")


def test_no_alloc_rejects_oversized_shapes(lib):
    """A shape whose workspace exceeds the fixed scratch array is refused with
    DF2_ERR_UNSUPPORTED and nothing runs.  The buffers are real and full-sized, so
    even a call that wrongly went ahead would stay in bounds."""
    P, D, V, K = 4096, 256, 2048, 1024
    need = lib.dflash2_unary_topk_workspace_size(P, D, V, K, 0)
    assert need > (8 << 20), need
    h = torch.zeros((P, D), dtype=torch.bfloat16, device="cuda")
    W = torch.zeros((V, D), dtype=torch.bfloat16, device="cuda")
    ids = torch.full((P, K), -7, dtype=torch.int32, device="cuda")
    vals = torch.empty((P, K), dtype=torch.float32, device="cuda")
    before = lib.dflash2_kernels_launched()
    rc = lib.dflash2_unary_topk_noalloc(_p(h), P, D, _p(W), V, K, 1.0, 0.0, None, 0, None, _p(ids), _p(vals),
                                        None, ct.c_void_p(torch.cuda.current_stream().cuda_stream))
    assert rc == 2 and lib.dflash2_status_string(rc) == b"DF2_ERR_UNSUPPORTED"
    assert lib.dflash2_kernels_launched() == before
    torch.cuda.synchronize()
    assert int(ids[0, 0].item()) == -7
