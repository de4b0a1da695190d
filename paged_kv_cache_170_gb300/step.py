"""A whole decode step recorded once as CUDA graphs and replayed.

One step is: copy-on-write block copies (when the step has any), slot lookup of
the new tokens, their K/V write, then split-context decode attention over every
sequence (the last three in one call when each sequence appends one token,
see ``DecodeStep``).  Launched one by one from Python, each call pays host-side argument
checks and a launch, and the GPU idles whenever the host falls behind; small
batches are then launch-bound.  Here the step's kernels are captured into two
CUDA graphs on first use: ``pre`` (copies, slots, write) and ``decode``.  A
replay launches them back to back with no host work in between.  Two graphs
rather than one so a caller can put CUDA events around the decode alone.

The graphs hold the device addresses of the step's tensors, so the caller
updates inputs in place (``q``, ``new_key`` / ``new_value``, the tables, ...)
and must not reallocate them.  Shapes are fixed at capture: a different batch
needs a new ``DecodeStep``.
"""
from __future__ import annotations

import copy
from types import SimpleNamespace
from typing import Optional

import torch

from . import ops


# The inputs a decode step consumes fresh every step (the pools stay resident).
STEP_INPUTS = ("q", "new_key", "new_value", "new_seq", "new_pos", "block_tables", "context_lens", "copy_pairs")


class PackedInputs:
    """A step's per-step inputs as views of one device buffer, mirrored by one
    pinned host buffer of the same layout, so that a step's inputs travel in a
    single host-to-device copy instead of one small copy per tensor (each small
    copy costs a few microseconds of fixed DMA latency on the GPU timeline).

    Construction moves ``inp``'s tensors named in ``names`` into the device
    buffer (replacing the attributes with views) and fills the host buffer with
    their current contents.  Build it before a ``DecodeStep``: the graphs then
    hold the packed addresses.  The caller writes the next step's inputs into
    ``host_views`` and calls ``upload()``.
    """

    def __init__(self, inp, names=STEP_INPUTS, align: int = 256):
        dev = inp.q.device
        layout, off = [], 0
        for n in names:
            t = getattr(inp, n)
            nbytes = t.numel() * t.element_size()
            layout.append((n, off, t.dtype, tuple(t.shape), nbytes))
            off += (nbytes + align - 1) // align * align
        self.nbytes = max(off, align)
        self.device = torch.zeros(self.nbytes, dtype=torch.uint8, device=dev)
        self.host = torch.zeros(self.nbytes, dtype=torch.uint8)
        if torch.cuda.is_available():
            self.host = self.host.pin_memory()
        self.host_views = {}
        for n, o, dtype, shape, nbytes in layout:
            t = getattr(inp, n)
            dv = self.device[o:o + nbytes].view(dtype).view(shape)
            hv = self.host[o:o + nbytes].view(dtype).view(shape)
            dv.copy_(t)
            hv.copy_(t.cpu())
            setattr(inp, n, dv)
            self.host_views[n] = hv

    def upload(self) -> None:
        """The host buffer into the device buffer: one copy on the current stream."""
        self.device.copy_(self.host, non_blocking=True)


def one_token_per_sequence(inp) -> bool:
    """True when the step appends one token to every sequence, at position
    context_lens - 1 (what pa_write_decode writes)."""
    S = inp.q.shape[0]
    if inp.new_seq.numel() != S or S == 0:
        return False
    seq = inp.new_seq.cpu().to(torch.int64)
    pos = inp.new_pos.cpu().to(torch.int64)
    lens = inp.context_lens.cpu().to(torch.int64)
    return bool(torch.equal(seq, torch.arange(S)) and torch.equal(pos, lens - 1) and (lens >= 1).all())


class DecodeStep:
    """The decode step of one set of resident inputs, as CUDA graphs.

    ``inp`` carries q, k_cache, v_cache, block_tables, context_lens, scale,
    new_key, new_value, new_seq, new_pos and copy_pairs (the layout of
    ``workloads.DecodeInputs``).  ``graphs=False`` launches the kernels one by
    one instead (same results, for comparison).  ``shared=True`` decodes with
    pa_decode_shared, reading each block that several sequences share once
    per group (the plan is built here from the tables).

    When every sequence appends exactly one token, at its last context
    position (``new_seq`` = 0 .. S-1, ``new_pos`` = context_lens - 1: a plain
    decode step), the write and the decode run as one call, pa_write_decode
    (slot lookup and write in one kernel; the decode starts launching while it
    runs); ``fused=False`` keeps the separate slot lookup, write and decode.
    The step's shape is checked here, at construction: later steps must keep
    it.
    """

    def __init__(self, inp, graphs: bool = True, shared: bool = False, fused: bool = True):
        self.inp = inp
        dev = inp.q.device
        S, Hq, D = inp.q.shape
        Hkv, B = inp.k_cache.shape[1], inp.k_cache.shape[2]
        self.out = torch.empty_like(inp.q)
        self.shared = shared
        self.fused = fused and not shared and one_token_per_sequence(inp)
        decode_launches = 1
        self.shared_kernels = []  # the shared decode's kernels, when it is not the plain decode
        if shared:
            # the plan follows the tables as the decode sees them; this step
            # only writes into private blocks, so it stays valid across replays
            self.plan = ops.share_plan(inp.block_tables, inp.context_lens, B, Hq, Hkv)
            self.plan_dev = self.plan.to(dev)
            self.plan_info = {k: v for k, v in ops.plan_fields(self.plan).items() if not k.endswith("_arr")}
            self.workspace = ops.new_shared_workspace(self.plan, S, Hq, Hkv, D, dev)
            if self.plan_info["num_shared_groups"] > 0:
                # the dense groups on the tensor cores, the other groups' blocks, then the merge
                f = ops.plan_fields(self.plan)
                cp, co = f["c_poff_arr"], f["c_opoff_arr"]
                self.shared_kernels = (["prefill_tc_kernel (dense groups)"] if self.plan_info["num_tc_items"] else []) + \
                    (["decode_shared_mma_kernel"] if int(cp[-1] - cp[0] + co[-1] - co[0]) > 0 else []) + \
                    ["merge_shared_kernel"]
                decode_launches = len(self.shared_kernels)
        else:
            self.workspace = ops.new_workspace(S, Hq, Hkv, D, dev)
        self.slots = torch.empty(inp.new_seq.numel(), dtype=torch.int64, device=dev)
        self.err = ops.new_error_word(dev)
        writes = 1 if self.fused else (2 if inp.new_seq.numel() else 0)
        self.launches_per_step = (1 if inp.copy_pairs.numel() else 0) + writes + decode_launches
        self.graphs = graphs
        # kernels before the decode: copy-on-write copies; slot lookup and write unless fused
        self.has_pre = bool(inp.copy_pairs.numel()) or (bool(inp.new_seq.numel()) and not self.fused)
        self._pre: Optional[torch.cuda.CUDAGraph] = None
        self._dec: Optional[torch.cuda.CUDAGraph] = None
        if graphs:
            # one eager pass first: the library sets its kernels' attributes and
            # caches device properties outside the capture
            self._run_pre()
            self._run_decode()
            torch.cuda.synchronize(dev)
            if self.has_pre:
                self._pre = torch.cuda.CUDAGraph()
                with torch.cuda.graph(self._pre):
                    self._run_pre()
            self._dec = torch.cuda.CUDAGraph()
            with torch.cuda.graph(self._dec):
                self._run_decode()

    def _run_pre(self):
        inp = self.inp
        if inp.copy_pairs.numel():
            ops.pa_copy_blocks(inp.k_cache, inp.v_cache, inp.copy_pairs, self.err)
        if inp.new_seq.numel() and not self.fused:
            ops.pa_slot_mapping(inp.block_tables, inp.new_seq, inp.new_pos, inp.k_cache.shape[2],
                                inp.k_cache.shape[0], self.slots, self.err)
            ops.pa_write_kv(inp.new_key, inp.new_value, inp.k_cache, inp.v_cache, self.slots, self.err)

    def _run_decode(self):
        inp = self.inp
        if self.shared:
            ops.pa_decode_shared(inp.q, inp.k_cache, inp.v_cache, inp.block_tables, inp.context_lens, inp.scale,
                                 self.plan, self.plan_dev, self.out, self.workspace, self.err)
        elif self.fused:
            ops.pa_write_decode(inp.q, inp.new_key, inp.new_value, inp.k_cache, inp.v_cache, inp.block_tables,
                                inp.context_lens, inp.scale, self.out, self.workspace, self.err)
        else:
            ops.pa_decode(inp.q, inp.k_cache, inp.v_cache, inp.block_tables, inp.context_lens, inp.scale, self.out,
                          self.workspace, self.err)

    def run(self, ev_decode_start=None, ev_decode_end=None) -> torch.Tensor:
        """Enqueue one step on the current stream; optional events bracket the
        decode.  Returns ``out`` (written when the stream reaches it)."""
        stream = torch.cuda.current_stream(self.inp.q.device)
        if self._pre is not None:
            self._pre.replay()
        elif self.has_pre:
            self._run_pre()
        if ev_decode_start is not None:
            ev_decode_start.record(stream)
        if self._dec is not None:
            self._dec.replay()
        else:
            self._run_decode()
        if ev_decode_end is not None:
            ev_decode_end.record(stream)
        return self.out


class StepPipeline:
    """Decode steps through host memory as a two-deep pipeline.

    Two step slots over the same K/V pools, each with its own packed inputs,
    output, pinned output mirror and graphs.  Step k runs in slot k mod 2: its
    inputs are uploaded on an upload stream once the slot's previous step has
    consumed them; the step runs on the caller's stream once that upload is in
    and the slot's previous output has been read back; its output is copied to
    the slot's pinned ``out_host`` on a download stream.  The uploads and
    downloads of one slot thus overlap the other slot's kernels, while the
    pools are written in step order on the one compute stream.  The caller
    writes the next step's inputs into ``slot.packed.host_views`` before
    ``step()`` and reads ``slot.out_host`` after ``slot.ev_down``.
    """

    def __init__(self, inp, graphs: bool = True, shared: bool = False, fused: bool = True):
        dev = inp.q.device
        self.device = dev
        self.slots = []
        for _ in range(2):
            si = copy.copy(inp)  # shares the pools; its per-step inputs are packed anew
            packed = PackedInputs(si)
            runner = DecodeStep(si, graphs=graphs, shared=shared, fused=fused)
            out_host = torch.empty(runner.out.shape, dtype=runner.out.dtype).pin_memory()
            plan_host = runner.plan.pin_memory() if shared else None
            self.slots.append(SimpleNamespace(inp=si, packed=packed, runner=runner, out_host=out_host,
                                              plan_host=plan_host, ev_up=torch.cuda.Event(),
                                              ev_done=torch.cuda.Event(), ev_down=torch.cuda.Event()))
        self.up_stream = torch.cuda.Stream(dev)
        self.down_stream = torch.cuda.Stream(dev)
        comp = torch.cuda.current_stream(dev)
        for sl in self.slots:  # nothing to wait for before the first two steps
            sl.ev_done.record(comp)
            sl.ev_down.record(comp)
        sl = self.slots[0]
        self.h2d_bytes = sl.packed.nbytes + (sl.plan_host.numel() * sl.plan_host.element_size() if shared else 0)
        self.d2h_bytes = sl.out_host.numel() * sl.out_host.element_size()
        self.k = 0

    def next_host_views(self) -> dict:
        """The pinned host views of the next step's inputs (``PackedInputs.host_views``
        of the slot ``step()`` uses next), once the upload of that slot's
        previous step has read them: the caller writes the step's inputs there,
        then calls ``step()``."""
        sl = self.slots[self.k % 2]
        sl.ev_up.synchronize()
        return sl.packed.host_views

    def next_host_buffer(self) -> torch.Tensor:
        """The same as one pinned uint8 buffer (every input in the packed
        layout of ``PackedInputs``): a caller that lays out a step's inputs
        itself writes them with one copy."""
        sl = self.slots[self.k % 2]
        sl.ev_up.synchronize()
        return sl.packed.host

    def step(self):
        """Enqueue the next step; returns its slot."""
        sl = self.slots[self.k % 2]
        comp = torch.cuda.current_stream(self.device)
        self.up_stream.wait_event(sl.ev_done)  # the slot's previous step has read its inputs
        with torch.cuda.stream(self.up_stream):
            sl.packed.upload()
            if sl.plan_host is not None:
                sl.runner.plan_dev.copy_(sl.plan_host, non_blocking=True)
            sl.ev_up.record(self.up_stream)
        comp.wait_event(sl.ev_up)
        comp.wait_event(sl.ev_down)  # the slot's previous output has been read back
        sl.runner.run()
        sl.ev_done.record(comp)
        self.down_stream.wait_event(sl.ev_done)
        with torch.cuda.stream(self.down_stream):
            sl.out_host.copy_(sl.runner.out, non_blocking=True)
            sl.ev_down.record(self.down_stream)
        self.k += 1
        return sl

    def drain(self) -> None:
        """Make the caller's stream wait for every download enqueued so far."""
        comp = torch.cuda.current_stream(self.device)
        for sl in self.slots:
            comp.wait_event(sl.ev_down)

