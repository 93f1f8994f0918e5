"""GB300-native partitioned mixed-precision ZeRO Adam step.

A thin Python binding of ``libzerostep.so`` (C ABI declared in
``include/zerostep.h``): the functions below only marshal arguments; every
step of the computation runs in the library's sm_103a kernels.  PyTorch is
used for device memory, streams and pinned host memory.

Entry points (same names as the C ABI):
  zero_partition_layout, zero_state_init, zero_workspace_bytes,
  zero_reduce_scatter_sum, zero_check_overflow, zero_grad_norm,
  zero_grad_norm_noalloc, zero_adam_step, zero_step_finalize,
  zero_step_fused, zero_reduce_scatter_accumulate,
  zero_step_fused_accumulated, zero_step_fused_buckets,
  zero_step_buckets_pass1, zero_step_buckets_norm, zero_step_buckets_pass2.
``ZeroStep`` owns the buffers of one simulated data-parallel group and runs
the fused step on them.
"""
from __future__ import annotations

import ctypes
from typing import List, Optional, Sequence, Tuple

import torch

from ._abi import (BF16, F16, MAX_WORLD, AdamCfg, Layout, StepState, ZeroError, check, lib)

HALF_REDUCE = 2  # added to F16 / BF16: reduce in the half type instead of fp32

__all__ = [
    "F16", "BF16", "MAX_WORLD", "AdamCfg", "Layout", "StepState", "ZeroError", "ZeroStep",
    "adam_cfg", "new_state", "new_workspace", "read_state", "state_field_ptr", "zero_partition_layout",
    "zero_state_init", "zero_workspace_bytes", "zero_reduce_scatter_sum", "zero_check_overflow",
    "zero_grad_norm", "zero_grad_norm_noalloc", "zero_adam_step", "zero_step_finalize", "zero_step_fused",
    "zero_reduce_scatter_accumulate", "zero_step_fused_accumulated", "zero_step_fused_buckets",
    "zero_step_buckets_pass1", "zero_step_buckets_norm", "zero_step_buckets_pass2",
    "host_empty",
]

_TORCH_DT = {F16: torch.float16, BF16: torch.bfloat16}


def _dtype_code(t: torch.Tensor) -> int:
    if t.dtype == torch.float16:
        return F16
    if t.dtype == torch.bfloat16:
        return BF16
    raise TypeError(f"half-precision tensor expected, got {t.dtype}")


def torch_dtype(code: int) -> torch.dtype:
    return _TORCH_DT[code]


def _dev_ptr(t: Optional[torch.Tensor]) -> Optional[int]:
    if t is None:
        return None
    if not t.is_cuda or not t.is_contiguous():
        raise ValueError("contiguous CUDA tensor expected")
    return t.data_ptr()


def _ptr_array(tensors: Sequence[torch.Tensor]):
    return (ctypes.c_void_p * len(tensors))(*[_dev_ptr(t) for t in tensors])


def _state_ptr(t: torch.Tensor) -> int:
    """A device tensor, or a pinned host tensor (offloaded optimizer state)."""
    if not t.is_contiguous() or not (t.is_cuda or t.is_pinned()):
        raise ValueError("contiguous CUDA or pinned host tensor expected")
    return t.data_ptr()


def _state_array(tensors: Sequence[torch.Tensor]):
    return (ctypes.c_void_p * len(tensors))(*[_state_ptr(t) for t in tensors])


def _grad_array(tensors: Sequence[torch.Tensor]):
    """Gradient buffers: CUDA tensors, or pinned host tensors that the
    kernels load directly over the host link."""
    return _state_array(tensors)


def _stream(stream) -> int:
    """The raw CUDA stream handle: the given stream, else torch's current one."""
    if stream is not None:
        return stream.cuda_stream
    raw = getattr(torch._C, "_cuda_getCurrentRawStream", None)
    if raw is not None:  # the handle itself, without building a Stream object
        return raw(torch.cuda.current_device())
    return torch.cuda.current_stream().cuda_stream


# ----------------------------------------------------------------- host helpers

def zero_partition_layout(numels: Sequence[int], world: int, align_elems: int = 64,
                          bucket_numel: int = 0) -> Tuple[Layout, List[int]]:
    """Step (a1).  Returns the layout and every tensor's flat offset."""
    n = len(numels)
    arr = (ctypes.c_int64 * max(n, 1))(*numels)
    offs = (ctypes.c_int64 * max(n, 1))()
    out = Layout()
    check("zero_partition_layout",
          lib().zero_partition_layout(n, arr, world, align_elems, bucket_numel, offs,
                                      ctypes.byref(out)))
    return out, list(offs[:n])


def zero_state_init(loss_scale: float = 1.0) -> StepState:
    s = StepState()
    check("zero_state_init", lib().zero_state_init(ctypes.byref(s), loss_scale))
    return s


def zero_workspace_bytes(layout: Optional[Layout] = None) -> int:
    """Workspace bytes of a step on `layout` (zero-fill it before first use),
    or with no layout the bytes zero_grad_norm needs."""
    n = lib().zero_workspace_bytes(ctypes.byref(layout) if layout is not None else None)
    if n == 0:
        raise ZeroError("zero_workspace_bytes", -1)
    return n


def new_workspace(layout: Optional[Layout] = None, device="cuda") -> torch.Tensor:
    """A zero-filled device workspace for steps on `layout` (or for
    zero_grad_norm with no layout)."""
    return torch.zeros(zero_workspace_bytes(layout), dtype=torch.uint8, device=device)


class _HostBlock:
    """One zero_host_alloc block, released when the last tensor over it is
    gone (the tensor keeps the buffer object alive, which keeps the block)."""

    def __init__(self, nbytes: int):
        p = ctypes.c_void_p()
        check("zero_host_alloc", lib().zero_host_alloc(nbytes, ctypes.byref(p)))
        self.ptr = p.value

    def __del__(self):
        if self.ptr:
            lib().zero_host_free(self.ptr)
            self.ptr = None


def host_empty(numel: int, dtype: torch.dtype) -> torch.Tensor:
    """A CPU tensor of `numel` elements in page-locked host memory from
    zero_host_alloc (contents undefined).  Copies from and to it run at the
    host link's full rate, and kernels may read or write it directly."""
    nbytes = int(numel) * torch.empty(0, dtype=dtype).element_size()
    if nbytes == 0:
        return torch.empty(0, dtype=dtype)
    block = _HostBlock(nbytes)
    buf = (ctypes.c_uint8 * nbytes).from_address(block.ptr)
    buf._block = block
    return torch.frombuffer(buf, dtype=torch.uint8).view(dtype)


def adam_cfg(lr: float = 1e-3, beta1: float = 0.9, beta2: float = 0.999, eps: float = 1e-8,
             weight_decay: float = 0.0, adamw: bool = True, bias_correction: bool = True,
             max_grad_norm: float = 0.0, dynamic_scale: bool = False, growth_interval: int = 1000,
             backoff: float = 0.5, growth: float = 2.0, min_scale: float = 1.0) -> AdamCfg:
    return AdamCfg(lr, beta1, beta2, eps, weight_decay, int(adamw), int(bias_correction),
                   max_grad_norm, int(dynamic_scale), growth_interval, backoff, growth, min_scale)


def new_state(loss_scale: float = 1.0, device="cuda") -> torch.Tensor:
    """A device-resident zero_step_state (192 bytes) in its initial state."""
    s = zero_state_init(loss_scale)
    host = torch.frombuffer(bytearray(bytes(s)), dtype=torch.uint8)
    return host.to(device)


def read_state(state: torch.Tensor) -> StepState:
    """Copy a device state to the host (synchronises with its stream)."""
    return StepState.from_buffer_copy(bytes(state.cpu().numpy().tobytes()))


def state_field_ptr(state: torch.Tensor, field: str) -> int:
    return state.data_ptr() + getattr(StepState, field).offset


# ----------------------------------------------------------------- device entry points

def _grad_code(grads, half_reduce: bool) -> int:
    return _dtype_code(grads[0]) | (HALF_REDUCE if half_reduce else 0)


def zero_reduce_scatter_sum(grads: Sequence[torch.Tensor], layout: Layout, g_out: torch.Tensor,
                            rank: int = -1, grads_are_slices: bool = False, stream=None,
                            half_reduce: bool = False) -> None:
    check("zero_reduce_scatter_sum",
          lib().zero_reduce_scatter_sum(_grad_array(grads), int(grads_are_slices),
                                        _grad_code(grads, half_reduce), ctypes.byref(layout),
                                        rank, _dev_ptr(g_out), _stream(stream)))


def zero_check_overflow(g: torch.Tensor, inv_scale: float, flag_ptr: int, stream=None) -> None:
    check("zero_check_overflow",
          lib().zero_check_overflow(_dev_ptr(g), g.numel(), inv_scale, flag_ptr, _stream(stream)))


def zero_grad_norm(g: torch.Tensor, inv_scale: float, sumsq_ptr: int, ws: torch.Tensor,
                   stream=None) -> None:
    check("zero_grad_norm",
          lib().zero_grad_norm(_dev_ptr(g), g.numel(), inv_scale, sumsq_ptr, _dev_ptr(ws),
                               ws.numel() * ws.element_size(), _stream(stream)))


def zero_grad_norm_noalloc(g: torch.Tensor, inv_scale: float, sumsq_ptr: int,
                           stream=None) -> None:
    """zero_grad_norm without a workspace: the partial sums live in a small
    library-owned device array (see include/zerostep.h)."""
    check("zero_grad_norm_noalloc",
          lib().zero_grad_norm_noalloc(_dev_ptr(g), g.numel(), inv_scale, sumsq_ptr,
                                       _stream(stream)))


def zero_adam_step(g: torch.Tensor, master: torch.Tensor, m: torch.Tensor, v: torch.Tensor,
                   half_out: torch.Tensor, cfg: AdamCfg, state: torch.Tensor, stream=None) -> None:
    check("zero_adam_step",
          lib().zero_adam_step(_dev_ptr(g), _dev_ptr(master), _dev_ptr(m), _dev_ptr(v),
                               _dev_ptr(half_out), _dtype_code(half_out), g.numel(),
                               ctypes.byref(cfg), _dev_ptr(state), _stream(stream)))


def zero_step_finalize(cfg: AdamCfg, state: torch.Tensor, flip_slot: bool = False,
                       stream=None) -> None:
    check("zero_step_finalize",
          lib().zero_step_finalize(ctypes.byref(cfg), _dev_ptr(state), int(flip_slot),
                                   _stream(stream)))


def zero_step_fused(grads: Sequence[torch.Tensor], layout: Layout,
                    master: Sequence[torch.Tensor], m: Sequence[torch.Tensor],
                    v: Sequence[torch.Tensor], params: Sequence[torch.Tensor], cfg: AdamCfg,
                    state: torch.Tensor, ws: torch.Tensor, rank: int = -1,
                    g_stage: Optional[torch.Tensor] = None, grads_are_slices: bool = False,
                    stream=None, half_reduce: bool = False) -> None:
    """The whole step (a2)-(a8).  master, m, v and params are the two
    ping-pong slots (the same tensor twice for an in-place clipped step);
    master, m and v may be pinned host tensors (offloaded state)."""
    check("zero_step_fused",
          lib().zero_step_fused(_grad_array(grads), int(grads_are_slices),
                                _grad_code(grads, half_reduce),
                                ctypes.byref(layout), rank, _state_array(master), _state_array(m),
                                _state_array(v), _ptr_array(params), _dev_ptr(g_stage),
                                ctypes.byref(cfg), _dev_ptr(state), _dev_ptr(ws),
                                ws.numel() * ws.element_size(), _stream(stream)))


def zero_step_fused_buckets(grads: Sequence[torch.Tensor], layout: Layout, first_bucket: int,
                            n_buckets: int, master: Sequence[torch.Tensor],
                            m: Sequence[torch.Tensor], v: Sequence[torch.Tensor],
                            params: Sequence[torch.Tensor], cfg: AdamCfg, state: torch.Tensor,
                            rank: int = -1, grads_are_slices: bool = False, stream=None,
                            half_reduce: bool = False) -> None:
    """Steps (a2)-(a7) of the one-pass step on buckets [first_bucket,
    first_bucket + n_buckets), without the commit; zero_step_finalize(cfg,
    state, flip_slot=True) commits once every bucket has been processed."""
    check("zero_step_fused_buckets",
          lib().zero_step_fused_buckets(_grad_array(grads), int(grads_are_slices),
                                        _grad_code(grads, half_reduce), ctypes.byref(layout),
                                        rank, first_bucket, n_buckets, _state_array(master),
                                        _state_array(m), _state_array(v), _ptr_array(params),
                                        ctypes.byref(cfg), _dev_ptr(state), _stream(stream)))


def zero_step_buckets_pass1(grads: Sequence[torch.Tensor], layout: Layout, first_bucket: int,
                            n_buckets: int, cfg: AdamCfg, state: torch.Tensor, ws: torch.Tensor,
                            rank: int = -1, g_stage: Optional[torch.Tensor] = None,
                            grads_are_slices: bool = False, stream=None,
                            half_reduce: bool = False) -> None:
    """First pass of the clipped step on buckets [first_bucket, first_bucket
    + n_buckets): reduce, unscale, flag, the squares into the workspace's
    tree (and the unscaled gradient into g_stage when given)."""
    check("zero_step_buckets_pass1",
          lib().zero_step_buckets_pass1(_grad_array(grads), int(grads_are_slices),
                                        _grad_code(grads, half_reduce), ctypes.byref(layout),
                                        rank, first_bucket, n_buckets, _dev_ptr(g_stage),
                                        ctypes.byref(cfg), _dev_ptr(state), _dev_ptr(ws),
                                        ws.numel() * ws.element_size(), _stream(stream)))


def zero_step_buckets_norm(layout: Layout, ws: torch.Tensor, rank: int = -1,
                           stream=None) -> None:
    """The clipped step's global sum of squares, after the first pass on
    every bucket and before the second pass on any."""
    check("zero_step_buckets_norm",
          lib().zero_step_buckets_norm(ctypes.byref(layout), rank, _dev_ptr(ws),
                                       ws.numel() * ws.element_size(), _stream(stream)))


def zero_step_buckets_pass2(grads: Optional[Sequence[torch.Tensor]], layout: Layout,
                            first_bucket: int, n_buckets: int, master: Sequence[torch.Tensor],
                            m: Sequence[torch.Tensor], v: Sequence[torch.Tensor],
                            params: Sequence[torch.Tensor], cfg: AdamCfg, state: torch.Tensor,
                            ws: torch.Tensor, rank: int = -1,
                            g_stage: Optional[torch.Tensor] = None, dtype: Optional[int] = None,
                            grads_are_slices: bool = False, stream=None,
                            half_reduce: bool = False) -> None:
    """Second pass of the clipped step on a range of buckets: clip, Adam,
    cast; the gradient is reduced again (grads) or read from g_stage."""
    if grads is not None:
        code = _grad_code(grads, half_reduce)
        garr = _grad_array(grads)
    else:
        code = (dtype if dtype is not None else _dtype_code(params[0])) | (
            HALF_REDUCE if half_reduce else 0)
        garr = None
    check("zero_step_buckets_pass2",
          lib().zero_step_buckets_pass2(garr, int(grads_are_slices), code, ctypes.byref(layout),
                                        rank, first_bucket, n_buckets, _state_array(master),
                                        _state_array(m), _state_array(v), _ptr_array(params),
                                        _dev_ptr(g_stage), ctypes.byref(cfg), _dev_ptr(state),
                                        _dev_ptr(ws), ws.numel() * ws.element_size(),
                                        _stream(stream)))


def zero_reduce_scatter_accumulate(grads: Sequence[torch.Tensor], layout: Layout,
                                   acc: torch.Tensor, add: bool, rank: int = -1,
                                   grads_are_slices: bool = False, stream=None,
                                   half_reduce: bool = False) -> None:
    """One micro-step of gradient accumulation: acc = (acc if add else 0) +
    the reduce-scatter sum of the ranks' half gradients."""
    check("zero_reduce_scatter_accumulate",
          lib().zero_reduce_scatter_accumulate(_grad_array(grads), int(grads_are_slices),
                                               _grad_code(grads, half_reduce),
                                               ctypes.byref(layout), rank,
                                               _dev_ptr(acc), int(add), _stream(stream)))


def zero_step_fused_accumulated(acc: torch.Tensor, dtype: int, layout: Layout,
                                master: Sequence[torch.Tensor], m: Sequence[torch.Tensor],
                                v: Sequence[torch.Tensor], params: Sequence[torch.Tensor],
                                cfg: AdamCfg, state: torch.Tensor, ws: torch.Tensor,
                                rank: int = -1, stream=None) -> None:
    """The step with the gradient taken from the fp32 accumulator."""
    check("zero_step_fused_accumulated",
          lib().zero_step_fused_accumulated(_dev_ptr(acc), dtype, ctypes.byref(layout), rank,
                                            _ptr_array(master), _ptr_array(m), _ptr_array(v),
                                            _ptr_array(params), ctypes.byref(cfg),
                                            _dev_ptr(state), _dev_ptr(ws),
                                            ws.numel() * ws.element_size(), _stream(stream)))


# ----------------------------------------------------------------- buffer owner

class ZeroStep:
    """The buffers of one simulated data-parallel group and its fused step.

    rank = -1 simulates every rank (state buffers span the padded flat
    vector); rank = r simulates rank r alone (state buffers hold r's owned
    elements).  Without clipping the master/m/v/params buffers are
    double-buffered so an overflow step can be skipped in one pass; with
    clipping they are updated in place and the reduced gradient is staged in
    fp32 between the two passes when that reads fewer bytes (N_d > 4).
    offload_state keeps master, m and v in page-locked host memory from
    zero_host_alloc (ZeRO-Offload style; the GPU reaches them over the host
    link).
    """

    def __init__(self, numels: Sequence[int], world: int, dtype: int, cfg: AdamCfg,
                 loss_scale: float = 1.0, rank: int = -1, bucket_numel: int = 0,
                 align_elems: int = 64, grads_are_slices: bool = False,
                 stage_grad: Optional[bool] = None, device="cuda", half_reduce: bool = False,
                 offload_state: bool = False):
        self.layout, self.offsets = zero_partition_layout(numels, world, align_elems, bucket_numel)
        self.world, self.dtype, self.cfg, self.rank = world, dtype, cfg, rank
        self.half_reduce = half_reduce
        self.grads_are_slices = grads_are_slices
        L = self.layout
        self.n_state = L.padded_numel if rank < 0 else L.owned_numel
        clip = cfg.max_grad_norm > 0
        hdt = torch_dtype(dtype)
        if offload_state and clip:
            raise ValueError("offloaded optimizer state supports the one-pass step (no clip)")
        f32 = dict(dtype=torch.float32, device=device)
        slots = 1 if clip else 2

        def state_buffer():
            if offload_state:
                return host_empty(self.n_state, torch.float32).zero_()
            return torch.zeros(self.n_state, **f32)

        self.master = [state_buffer() for _ in range(slots)]
        self.m = [state_buffer() for _ in range(slots)]
        self.v = [state_buffer() for _ in range(slots)]
        self.params = [torch.zeros(L.padded_numel, dtype=hdt, device=device) for _ in range(slots)]
        if slots == 1:
            for lst in (self.master, self.m, self.v, self.params):
                lst.append(lst[0])
        if stage_grad is None:
            stage_grad = clip and world > 4
        self.g_stage = torch.empty(self.n_state, **f32) if (clip and stage_grad) else None
        self.state = new_state(loss_scale, device)
        self.ws = new_workspace(self.layout, device)

    def segments(self, r: int) -> List[Tuple[int, int]]:
        """(flat start, length) of the ranges rank r owns, in r's element order."""
        L = self.layout
        if L.padded_numel == 0:
            return []
        if L.bucket_numel == 0:
            return [(r * L.owned_numel, L.owned_numel)]
        segs = [(b * L.bucket_numel + r * L.slice_numel, L.slice_numel)
                for b in range(L.num_buckets - 1)]
        segs.append(((L.num_buckets - 1) * L.bucket_numel + r * L.last_slice_numel,
                     L.last_slice_numel))
        return segs

    def grad_numel(self) -> int:
        """Elements of each rank's gradient buffer."""
        return self.layout.owned_numel if self.grads_are_slices else self.layout.padded_numel

    def _slots(self):
        """The ctypes arrays of the ping-pong slots, built once per set of
        slot tensors (the tensors are owned by this object)."""
        key = tuple(map(id, (*self.master, *self.m, *self.v, *self.params)))
        if getattr(self, "_slots_key", None) != key:
            self._slot_arrays = (_state_array(self.master), _state_array(self.m),
                                 _state_array(self.v), _ptr_array(self.params))
            self._slots_key = key
        return self._slot_arrays

    def step(self, grads: Sequence[torch.Tensor], stream=None) -> None:
        """The whole step (zero_step_fused) on this group's buffers."""
        w, m, v, p = self._slots()
        ws = self.ws
        check("zero_step_fused",
              lib().zero_step_fused(_grad_array(grads), int(self.grads_are_slices),
                                    _grad_code(grads, self.half_reduce), ctypes.byref(self.layout),
                                    self.rank, w, m, v, p, _dev_ptr(self.g_stage),
                                    ctypes.byref(self.cfg), _dev_ptr(self.state), _dev_ptr(ws),
                                    ws.numel() * ws.element_size(), _stream(stream)))

    def step_buckets(self, grads: Sequence[torch.Tensor], first_bucket: int, n_buckets: int,
                     stream=None) -> None:
        """The one-pass step on a range of buckets, without the commit."""
        zero_step_fused_buckets(grads, self.layout, first_bucket, n_buckets, self.master,
                                self.m, self.v, self.params, self.cfg, self.state, self.rank,
                                self.grads_are_slices, stream, self.half_reduce)

    def pass1_buckets(self, grads: Sequence[torch.Tensor], first_bucket: int, n_buckets: int,
                      stream=None) -> None:
        """The clipped step's first pass on a range of buckets."""
        zero_step_buckets_pass1(grads, self.layout, first_bucket, n_buckets, self.cfg,
                                self.state, self.ws, self.rank, self.g_stage,
                                self.grads_are_slices, stream, self.half_reduce)

    def norm_buckets(self, stream=None) -> None:
        """The clipped step's global norm, between the two passes."""
        zero_step_buckets_norm(self.layout, self.ws, self.rank, stream)

    def pass2_buckets(self, grads: Optional[Sequence[torch.Tensor]], first_bucket: int,
                      n_buckets: int, stream=None) -> None:
        """The clipped step's second pass on a range of buckets (the gradient
        from the stage when the group keeps one, else reduced again from
        grads)."""
        zero_step_buckets_pass2(None if self.g_stage is not None else grads, self.layout,
                                first_bucket, n_buckets, self.master, self.m, self.v,
                                self.params, self.cfg, self.state, self.ws, self.rank,
                                self.g_stage, self.dtype, self.grads_are_slices, stream,
                                self.half_reduce)

    def commit(self, stream=None) -> None:
        """End a step run bucket by bucket: commit, or skip on NaN/Inf."""
        zero_step_finalize(self.cfg, self.state, True, stream)

    def accumulate(self, grads: Sequence[torch.Tensor], add: bool, stream=None) -> None:
        """One micro-step into the group's fp32 gradient accumulator (allocated
        on first use); add=False starts a new accumulation."""
        if getattr(self, "acc", None) is None:
            self.acc = torch.empty(self.n_state, dtype=torch.float32, device=self.state.device)
        zero_reduce_scatter_accumulate(grads, self.layout, self.acc, add, self.rank,
                                       self.grads_are_slices, stream, self.half_reduce)

    def step_accumulated(self, stream=None) -> None:
        """The step from the accumulated gradient."""
        zero_step_fused_accumulated(self.acc, self.dtype, self.layout, self.master, self.m,
                                    self.v, self.params, self.cfg, self.state, self.ws, self.rank,
                                    stream)

    def step_from_host(self, host_grads: Sequence[torch.Tensor],
                       device_grads: Optional[Sequence[torch.Tensor]] = None, stream=None,
                       micro_steps: int = 1) -> StepState:
        """End to end from each rank's gradient in page-locked host memory:
        run the step and read the step state back to the host.  Without
        device_grads the step's kernels load the gradients straight from the
        host buffers over the host link; with device_grads each gradient is
        first copied into its device buffer by the copy engines.  With
        micro_steps > 1 the same host buffers stand for every micro-step, each
        reduced into the fp32 accumulator before the step."""
        s = stream if stream is not None else torch.cuda.current_stream()
        if getattr(self, "_state_host", None) is None:
            self._state_host = host_empty(ctypes.sizeof(StepState), torch.uint8)
        with torch.cuda.stream(s):
            for k in range(micro_steps):
                grads = host_grads
                if device_grads is not None:
                    for h, d in zip(host_grads, device_grads):
                        d.copy_(h, non_blocking=True)
                    grads = device_grads
                if micro_steps > 1:
                    self.accumulate(grads, k > 0, s)
            if micro_steps > 1:
                self.step_accumulated(s)
            else:
                self.step(grads, s)
            self._state_host.copy_(self.state, non_blocking=True)
        s.synchronize()
        return StepState.from_buffer_copy(bytes(self._state_host.numpy().tobytes()))

    def read_state(self) -> StepState:
        return read_state(self.state)

    def current(self):
        """(master, m, v, params) of the slot holding the current state."""
        c = self.read_state().cur
        return self.master[c], self.m[c], self.v[c], self.params[c]
