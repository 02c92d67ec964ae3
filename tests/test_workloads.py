"""Host-side workload logic (no GPU): the synthetic stacks' shapes and which
layers share an input, as the benchmark and the grouped projections use them."""
import importlib.util
import os

import pytest

from rank_gradient_sketching_philox_gb300 import synth

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _bench():
    spec = importlib.util.spec_from_file_location("bench_module", os.path.join(ROOT, "bench.py"))
    mod = importlib.util.module_from_spec(spec)
    spec.loader.exec_module(mod)
    return mod


def test_qwen3_8b_stack_shapes():
    """252 linears; the sums of output and input widths of the 8B shape."""
    wl = synth.WORKLOADS["qwen3-8b-stack"]
    assert len(wl.layers) == 252
    assert sum(d for _, d, _ in wl.layers) == 1_400_832
    assert sum(k for _, _, k in wl.layers) == 1_327_104
    assert wl.weights == 6_945_767_424
    assert wl.microbatches == 8


def test_input_groups_of_a_block():
    """q, k and v read one input, gate and up another; o and down their own.
    Every layer is in exactly one group and a group's layers have one k."""
    layers = synth.qwen3_stack(2, 4096, 1024, 12288)
    groups = synth.input_groups(layers)
    assert groups == [[0, 1, 2], [3], [4, 5], [6], [7, 8, 9], [10], [11, 12], [13]]
    assert sorted(li for g in groups for li in g) == list(range(len(layers)))
    for g in groups:
        assert len({layers[li][2] for li in g}) == 1


@pytest.mark.parametrize("name", sorted(synth.WORKLOADS))
def test_input_groups_cover_every_workload(name):
    layers = synth.WORKLOADS[name].layers
    groups = synth.input_groups(layers)
    assert sorted(li for g in groups for li in g) == list(range(len(layers)))
    assert all(len(g) * 64 <= 256 for g in groups)  # a group's rank m r fits one projection call


def test_bench_groups_follow_the_flag_and_rank():
    bench = _bench()
    wl = synth.WORKLOADS["qwen3-8b-stack"]
    shared = bench.workload_groups(wl, 64, False)
    assert len(shared) == 36 * 4
    assert bench.workload_groups(wl, 64, True) == [[li] for li in range(252)]
    assert bench.workload_groups(wl, 20, False) == [[li] for li in range(252)]  # members must start 16-byte aligned
    assert "one X each" in bench.input_note(shared)
    assert bench.input_note([[0], [1]]) == "every layer reads its own X"
