"""A whole fwd+bwd step captured as a CUDA graph and replayed.

cfa_forward, cfa_backward_preprocess and cfa_backward do no host
synchronisation and no allocation, and fork / join their second stream with
events, so a caller can capture them into a CUDA graph (the benchmark times
the step that way).  The replays must give bitwise the outputs of the same
calls launched one by one, for the bf16 and the q8_0 prefix, and leave the
device status clean.
"""
import pytest
import torch

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("name", ["qwen3_1p7b", "tiny"])
@pytest.mark.parametrize("mode", ["bf16", "q8_product", "q8_export"])
def test_graph_replay_equals_stream_launches(name, mode):
    import bench
    import synth
    dev = torch.device("cuda", 0)
    w = synth.workload(name, seed=0)
    if mode != "bf16":
        w.prefix_dtype = synth.PREFIX_Q8_0
    case = bench.AttnStep(w, dev, 0, "export" if mode == "q8_export" else "product")
    for _ in range(2):
        case.step()
    torch.cuda.synchronize()
    case.check_status()
    ref = [t.clone() for t in case.outputs()]
    for t in case.outputs():
        t.fill_(0)
    case.capture()
    for t in case.outputs():
        t.fill_(0)
    for _ in range(3):
        case.replay()
    torch.cuda.synchronize()
    case.check_status()
    for a, b in zip(ref, case.outputs()):
        assert torch.equal(a, b)


def test_pipelined_end_to_end_reads_back_each_steps_outputs():
    """The benchmark's end-to-end loop: inputs copied in on one stream while
    the previous step runs, outputs copied out on another while the next one
    runs, two buffer sets alternating.  The outputs read back to the host are
    bitwise those of a step launched on its own (the same inputs every step),
    whichever buffer set the last step used."""
    import bench
    import synth
    dev = torch.device("cuda", 0)
    w = synth.workload("qwen3_1p7b", seed=0)
    case = bench.AttnStep(w, dev, 0, "product")
    case.step()
    torch.cuda.synchronize()
    ref = [t.cpu() for t in case.outputs()]
    pin = {k: case.host[k].pin_memory() for k in case.names}
    flush = bench.L2Flush(dev)
    for steps in (4, 5):
        outs_h = [torch.empty(t.shape, dtype=t.dtype, pin_memory=True) for t in ref]
        ms = bench.e2e_pipelined(case, pin, outs_h, steps, flush, dev)
        assert ms > 0
        for a, b in zip(ref, outs_h):
            assert torch.equal(a, b)
