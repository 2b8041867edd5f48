"""Host-side helpers of bench.py on CPU: the packing of a step's inputs into
one host buffer and one device buffer for the end-to-end timing."""
import torch

import bench
from learned_sparse_attention_gb300 import workloads as W


def test_pack_step_inputs_round_trip():
    spec = W.named_spec("tiny_bf16")
    wl = W.make_workload(spec, device=torch.device("cpu"))
    host_buf, dev_buf, views = bench.pack_step_inputs(wl.t, bench.STEP_INPUTS, "cpu", pin=False)
    base = dev_buf.data_ptr()
    # nothing is set before the one copy
    dev_buf.zero_()
    dev_buf.copy_(host_buf)
    seen = []
    for k in bench.STEP_INPUTS:
        v, src = views[k], wl.t[k]
        assert v.dtype == src.dtype and v.shape == src.shape and v.is_contiguous()
        assert (v.data_ptr() - base) % 256 == 0
        assert torch.equal(v.reshape(-1).view(torch.uint8), src.contiguous().reshape(-1).view(torch.uint8))
        seen.append((v.data_ptr() - base, v.numel() * v.element_size()))
    # slots do not overlap
    seen.sort()
    for (a, na), (b, _) in zip(seen, seen[1:]):
        assert a + na <= b
    # tensors that are not step inputs are passed through unchanged
    for k, v in wl.t.items():
        if k not in bench.STEP_INPUTS:
            assert views[k] is v
