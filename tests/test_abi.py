"""The C-ABI library without a GPU: it loads, exports every entry point the
header declares, sizes workspaces, and rejects bad arguments on the host
before launching anything (no call here reaches a kernel)."""
import ctypes
import os
import re

import pytest

from rank_gradient_sketching_philox_gb300 import binding

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "sketch.h")


@pytest.fixture(scope="module")
def lib():
    import __graft_entry__ as g
    g.build()
    return binding.lib()


def declared_functions():
    text = open(HEADER).read()
    return sorted(set(re.findall(r"SKETCH_API\s+[\w\s\*]+?\b(sketch_\w+)\s*\(", text)))


def test_header_declares_the_path():
    names = declared_functions()
    for required in ("sketch_sample_projection", "sketch_project_inputs", "sketch_accumulate",
                     "sketch_apply_update_normsgd", "sketch_apply_update_sgd",
                     "sketch_workspace_bytes", "sketch_read_device_errors",
                     "sketch_status_string", "sketch_last_error"):
        assert required in names


def test_library_exports_every_declared_symbol(lib):
    for name in declared_functions():
        assert hasattr(lib, name), name
    assert set(declared_functions()) <= set(binding.EXPORTS) | set(declared_functions())


def test_status_strings(lib):
    for st in range(5):
        assert lib.sketch_status_string(st)
    assert lib.sketch_status_string(99) == b"unknown status"


def test_workspace_sizes(lib):
    ws = binding.workspace_bytes
    # FP16 high/low parts of C and P, their fp32 row norms, the split's scales
    # (one per row of C, one per 128 rows of P: 32 floats in a 256-byte
    # block), two 256-byte counters and the exact-path tags: per 128 x 128
    # tile and epilogue warp a count byte and room for 128 2-byte tags
    tiles = 32 * 32
    queue = tiles * 16 * (1 + 128 * 2)
    assert ws(binding.OP_UPDATE_SGD, 0, 4096, 4096, 64) == (4 * (4096 + 4096) * 64 + 4 * (4096 + 4096)
                                                           + 4 * 4096 + 256 + 2 * 256 + queue)
    a = ws(binding.OP_UPDATE_NORMSGD, 0, 4096, 4096, 64)
    b = ws(binding.OP_UPDATE_NORMSGD, 0, 8192, 4096, 64)
    c = ws(binding.OP_UPDATE_NORMSGD, 0, 4096, 4096, 128)
    assert 0 < a < b and a < c
    assert ws(binding.OP_SAMPLE_PROJECTION, 0, 0, 4096, 64) > 64 * 64 * 4
    assert ws(binding.OP_UPDATE_NORMSGD, 0, 4096, 4096, 0) == 0     # invalid r
    assert ws(binding.OP_UPDATE_NORMSGD, 0, 4096, 4096, 257) == 0   # invalid r


def _call(fn, *args):
    return getattr(binding.lib(), fn)(*args)


NULL = None


@pytest.mark.parametrize("args,status,msg", [
    # (T, k, ld_x, r, ld_xp)
    ((0, 64, 64, 8, 8), binding.ERR_INVALID_ARG, "T="),
    ((16, 60, 64, 8, 8), binding.ERR_INVALID_ARG, "k=60"),
    ((16, 64, 60, 8, 8), binding.ERR_INVALID_ARG, "ld_x"),
    ((16, 64, 72, 0, 8), binding.ERR_INVALID_ARG, "r=0"),
    ((16, 64, 72, 300, 304), binding.ERR_INVALID_ARG, "r=300"),
    ((16, 64, 64, 8, 4), binding.ERR_INVALID_ARG, "ld_xp"),
    ((16, 64, 64, 8, 8), binding.ERR_INVALID_ARG, "X is NULL"),
])
def test_project_inputs_argument_errors(lib, args, status, msg):
    T, k, ld_x, r, ld_xp = args
    st = lib.sketch_project_inputs(NULL, T, k, ld_x, NULL, r, NULL, ld_xp, NULL, 0, NULL)
    assert st == status
    assert msg in lib.sketch_last_error().decode()


def test_accumulate_argument_errors(lib):
    assert lib.sketch_accumulate(NULL, 16, 0, 8, NULL, 8, 8, NULL, 1, NULL, 0, NULL) == binding.ERR_INVALID_ARG
    assert b"d=" in lib.sketch_last_error()
    assert lib.sketch_accumulate(NULL, 16, 10, 10, NULL, 8, 8, NULL, 1, NULL, 0, NULL) == binding.ERR_INVALID_ARG
    assert b"ld_d" in lib.sketch_last_error()
    assert lib.sketch_accumulate(NULL, 16, 10, 16, NULL, 8, 8, NULL, 1, NULL, 0, NULL) == binding.ERR_INVALID_ARG
    assert b"D is NULL" in lib.sketch_last_error()


def test_update_argument_errors(lib):
    st = lib.sketch_apply_update_normsgd(NULL, 8, 12, 16, NULL, NULL, 4, 1e-3, 0, 0, 0, NULL, NULL,
                                         NULL, NULL, 0, NULL)
    assert st == binding.ERR_INVALID_ARG and b"k=12" in lib.sketch_last_error()
    st = lib.sketch_apply_update_sgd(NULL, 8, 16, 16, NULL, NULL, 4, 1e-3, 0, 0, 0, NULL, NULL, 0, NULL)
    assert st == binding.ERR_INVALID_ARG and b"W is NULL" in lib.sketch_last_error()


def test_sample_projection_argument_errors(lib):
    st = lib.sketch_sample_projection(5, 0, 0, 0, 64, 8, NULL, NULL, NULL, 0, NULL)
    assert st == binding.ERR_INVALID_ARG and b"kind" in lib.sketch_last_error()
    st = lib.sketch_sample_projection(0, 0, 0, 0, 64, 8, NULL, NULL, NULL, 0, NULL)
    assert st == binding.ERR_INVALID_ARG and b"P is NULL" in lib.sketch_last_error()
    st = lib.sketch_sample_projection(1, 0, 0, 0, 63, 8, NULL, NULL, NULL, 0, NULL)
    assert st == binding.ERR_INVALID_ARG and b"k=63" in lib.sketch_last_error()


def test_read_device_errors_needs_output(lib):
    assert lib.sketch_read_device_errors(NULL, NULL) == binding.ERR_INVALID_ARG
    assert lib.sketch_read_exact_count(NULL, NULL) == binding.ERR_INVALID_ARG


def test_binding_refuses_cpu_tensors(lib):
    import torch
    X = torch.zeros(4, 8, dtype=torch.bfloat16)
    with pytest.raises(ValueError):
        binding.project_inputs(X, torch.zeros(8, 2), torch.zeros(4, 2, dtype=torch.bfloat16))


def test_launch_counter_ignores_rejected_calls(lib):
    """The launch counter moves only when a kernel is launched: a call that
    fails validation on the host launches nothing."""
    before = binding.kernel_launches()
    st = _call("sketch_project_inputs", NULL, 16, 60, 64, NULL, 8, NULL, 8, NULL, 0, NULL)
    assert st == binding.ERR_INVALID_ARG
    assert binding.kernel_launches() == before >= 0


def test_projection_split_sizes(lib):
    assert binding.projection_split_elems(4096, 64) == 2 * 64 * 4096
    assert binding.projection_split_elems(4096, 20) == 2 * 32 * 4096   # r padded to 16
    assert binding.projection_split_elems(60, 8) == 0                  # k not a multiple of 8
    assert binding.projection_split_elems(64, 257) == 0


def test_split_and_project_reject_missing_pointers(lib):
    before = binding.kernel_launches()
    probs = (binding.SplitProblem * 1)(binding.SplitProblem(None, 64, None))
    assert _call("sketch_split_projection_batched", 1, probs, 8, NULL) == binding.ERR_INVALID_ARG
    pp = (binding.ProjectProblem * 1)(binding.ProjectProblem(1 << 20, 16, 64, 64, None, 1 << 21, 8, None))
    assert _call("sketch_project_inputs_batched", 1, pp, 8, NULL, 0, NULL) == binding.ERR_INVALID_ARG
    assert "P_split" in binding.lib().sketch_last_error().decode()
    assert binding.kernel_launches() == before


def test_policy_sync_payload_is_the_factor_and_seed():
    import torch
    from rank_gradient_sketching_philox_gb300 import policy_sync
    C = torch.arange(12, dtype=torch.float32).view(4, 3)
    msg = policy_sync.message(C, 0.5, 7, 2, 5)
    assert msg.U is C and (msg.alpha_eta, msg.seed, msg.layer, msg.step) == (0.5, 7, 2, 5)  # nothing computed
    with pytest.raises(TypeError):
        policy_sync.message(C.double(), 0.5, 7, 2, 5)
    assert policy_sync.payload_bytes(4096, 64) == 4 * 4096 * 64 + 20       # vs 2*4096*4096 of BF16 W


def test_fp32_xp_needs_room_for_the_pair(lib):
    """The fp32-accurate XP form needs ld_xp >= 2 * round16(r)."""
    before = binding.kernel_launches()
    pp = (binding.ProjectProblem * 1)(binding.ProjectProblem(1 << 20, 16, 64, 64, 1 << 21, 1 << 22, 24, None))
    assert _call("sketch_project_inputs_fp32xp_batched", 1, pp, 8, NULL, 0, NULL) == binding.ERR_INVALID_ARG
    assert "ld_xp" in binding.lib().sketch_last_error().decode()
    ap = (binding.AccumulateProblem * 1)(binding.AccumulateProblem(1 << 20, 16, 64, 64, 1 << 21, 24, 1 << 22))
    assert _call("sketch_accumulate_fp32xp_batched", 1, ap, 8, 1, NULL, 0, NULL) == binding.ERR_INVALID_ARG
    assert binding.kernel_launches() == before
    assert binding.xp_split_cols(64) == 128 and binding.xp_split_cols(20) == 64


def test_grouped_split_rejects_bad_groups(lib):
    """Grouped splits: 1 <= m <= 16, m r <= 256, r a multiple of 8 when m > 1,
    every pointer present; rejected on the host with no launch."""
    before = binding.kernel_launches()
    ptrs = (ctypes.c_void_p * 3)(1 << 20, 1 << 21, 1 << 22)
    P = ctypes.cast(ptrs, ctypes.c_void_p)

    def grouped(m, k, r, split=1 << 23, p=P):
        g = (binding.SplitGroup * 1)(binding.SplitGroup(p, m, k, split))
        return _call("sketch_split_projection_grouped", 1, g, r, NULL)

    assert grouped(0, 64, 64) == binding.ERR_INVALID_ARG
    assert grouped(17, 64, 8) == binding.ERR_INVALID_ARG
    assert grouped(3, 64, 96) == binding.ERR_INVALID_ARG        # 3 * 96 > 256
    assert "256" in binding.lib().sketch_last_error().decode()
    assert grouped(3, 64, 20) == binding.ERR_INVALID_ARG        # members would start off 16-byte boundaries
    assert grouped(3, 60, 64) == binding.ERR_INVALID_ARG        # k not a multiple of 8
    assert grouped(3, 64, 64, split=None) == binding.ERR_INVALID_ARG
    assert grouped(3, 64, 64, p=None) == binding.ERR_INVALID_ARG
    assert binding.kernel_launches() == before
