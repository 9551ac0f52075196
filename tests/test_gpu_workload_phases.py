"""Concurrent phases of a workload step give the results of the same ops run
one after another on one stream.

A workload may run the ops of a phase on side streams (the weight and the
activation quantizer of a linear layer share no data).  The step with its
phases and the step with the phases removed must write bit-identical outputs;
a phase whose ops shared data would race and differ.
"""
import pytest
import torch

from learnable_scale_fake_gb300 import workloads

pytestmark = pytest.mark.gpu


def _outputs(wl):
    return {k: v.clone() for k, v in wl.outputs.items()}


@pytest.mark.parametrize("name", ["nvfp4_wa", "nvfp4_wa_fused"])
def test_phases_match_sequential(name):
    dev = torch.device("cuda", 0)
    wl = workloads.BUILDERS[name](dev)
    assert wl.phases, "the workload declares concurrent phases"
    st = torch.cuda.Stream(dev)
    st.wait_stream(torch.cuda.current_stream())
    for _ in range(3):  # several steps: the side streams are reused
        wl.step(st)
    torch.cuda.synchronize()
    concurrent = _outputs(wl)
    phases, wl.phases = wl.phases, None
    try:
        for o in wl.outputs.values():
            o.zero_()
        torch.cuda.synchronize()
        wl.step(st)
        torch.cuda.synchronize()
    finally:
        wl.phases = phases
    for k, v in wl.outputs.items():
        a, b = concurrent[k], v
        assert torch.equal(a.view(torch.uint8), b.view(torch.uint8)), f"{k} differs"
