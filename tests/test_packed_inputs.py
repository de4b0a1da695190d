"""PackedInputs (host only): the per-step inputs become views of one buffer
with their contents intact, each 256-byte aligned, empty tensors included,
and the host mirror holds the same bytes."""
import torch

from paged_kv_cache_170_gb300 import workloads as W
from paged_kv_cache_170_gb300.step import STEP_INPUTS, PackedInputs


def test_packed_views_keep_contents_and_alignment():
    inp = W.make_inputs(W.WORKLOADS["tiny"], 0)
    before = {n: getattr(inp, n).clone() for n in STEP_INPUTS}
    packed = PackedInputs(inp)
    base = packed.device.data_ptr()
    end = base + packed.nbytes
    for n in STEP_INPUTS:
        t = getattr(inp, n)
        assert torch.equal(t, before[n]) and t.dtype == before[n].dtype and t.shape == before[n].shape
        assert torch.equal(packed.host_views[n], before[n])
        if t.numel():
            assert (t.data_ptr() - base) % 256 == 0 and base <= t.data_ptr() and t.data_ptr() + t.nbytes <= end
    assert inp.copy_pairs.numel() == 0  # the tiny workload copies no block: an empty view
    # the host mirror is the device buffer's image byte for byte
    assert torch.equal(packed.host, packed.device.cpu())


def test_upload_moves_new_inputs_in_one_copy():
    inp = W.make_inputs(W.WORKLOADS["tiny"], 0)
    packed = PackedInputs(inp)
    packed.host_views["q"].mul_(2)
    packed.host_views["context_lens"].add_(1)
    packed.upload()
    assert torch.equal(inp.q, packed.host_views["q"])
    assert torch.equal(inp.context_lens, packed.host_views["context_lens"])
