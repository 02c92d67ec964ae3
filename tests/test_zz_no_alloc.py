"""The allocation-free normalized-SGD update, called through the C ABI.

sketch_apply_update_normsgd_noalloc exists for callers that cannot allocate
device memory (a plugin handed only its input and output buffers, or a process
whose device memory is already given to another pool).  It must produce what
sketch_apply_update_normsgd produces with a caller-provided workspace.  This
file is named to be collected last, so a run that stops at the first failure
has run every other test before it; it also passes on its own in a fresh
process, where its first call sets up the scratch array.
"""
import ctypes

import pytest
import torch

from rank_gradient_sketching_philox_gb300 import binding, synth


pytestmark = pytest.mark.gpu

DEV = torch.device("cuda:0")


def _p(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


@pytest.fixture(scope="module")
def lib():
    import __graft_entry__ as g
    g.build()
    return binding.lib()


def test_noalloc_update_matches_workspace_update_on_two_calls(lib):
    d, k, r = 1024, 2048, 64
    W0 = synth.layer_weight(d, k, 6, device=DEV)
    Wa, Wb = W0.clone(), W0.clone()
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    na = torch.zeros(1, dtype=torch.float64, device=DEV)
    nb = torch.zeros(1, dtype=torch.float64, device=DEV)
    sa = torch.full((1,), -1, dtype=torch.int32, device=DEV)
    sb = torch.full((1,), -1, dtype=torch.int32, device=DEV)
    for step in (0, 1):  # two calls in a row: refreshed projection, carried ||W||^2
        P = torch.empty(k, r, dtype=torch.float32, device=DEV)
        binding.sample_projection(binding.PROJ_GAUSSIAN_QR, 5, 6, step, P)
        C = torch.randn(d, r, generator=torch.Generator(device=DEV).manual_seed(step), device=DEV)
        nbytes = binding.workspace_bytes(binding.OP_UPDATE_NORMSGD, 0, d, k, r)
        ws = torch.empty(nbytes, dtype=torch.uint8, device=DEV)
        st = lib.sketch_apply_update_normsgd(_p(Wa), d, k, k, _p(C), _p(P), r, 1e-3, 5, 6, step,
                                             _p(na) if step else None, _p(na), _p(sa), _p(ws), nbytes,
                                             stream)
        assert st == binding.OK, lib.sketch_last_error()
        st = lib.sketch_apply_update_normsgd_noalloc(_p(Wb), d, k, k, _p(C), _p(P), r, 1e-3, 5, 6, step,
                                                     _p(nb) if step else None, _p(nb), _p(sb), stream)
        assert st == binding.OK, lib.sketch_last_error()
        torch.cuda.synchronize()
        assert int(sa.item()) == 0 and int(sb.item()) == 0
        # the same computation in the same order: identical bits, identical norm
        assert torch.equal(Wb, Wa)
        assert nb.item() == na.item()
    assert not torch.equal(Wb, W0)
    assert binding.read_device_errors() == 0


def test_noalloc_update_rejects_layers_beyond_its_scratch(lib):
    d, k, r = 28672, 8192, 256
    need = binding.workspace_bytes(binding.OP_UPDATE_NORMSGD, 0, d, k, r)
    assert need > lib.sketch_noalloc_scratch_bytes()
    W = torch.zeros(d, k, dtype=torch.bfloat16, device=DEV)
    C = torch.zeros(d, r, dtype=torch.float32, device=DEV)
    P = torch.zeros(k, r, dtype=torch.float32, device=DEV)
    st = lib.sketch_apply_update_normsgd_noalloc(_p(W), d, k, k, _p(C), _p(P), r, 1e-3, 0, 0, 0, None, None,
                                                 None, None)
    assert st == binding.ERR_WORKSPACE
    assert b"fixed" in lib.sketch_last_error()
