"""GB300-native video sparse attention (VSA) forward.

Thin Python binding over the C ABI in ``include/vsa.h`` (``libvsa.so``, built
in-tree by ``block_sparse_video_gb300.build``). The functions keep the C names
and only marshal arguments: torch tensors are used for device memory and
streams; every step of the computation runs in the library's CUDA kernels.
If the library has not been built, the first call into it raises: there is
no fallback path.
"""
from __future__ import annotations

import ctypes
import os
import re

import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libvsa.so")
HEADER_PATH = os.path.join(os.path.dirname(_HERE), "include", "vsa.h")

VSA_OK = 0
VSA_ERR_INVALID_ARG = 1
VSA_ERR_UNSUPPORTED = 2
VSA_ERR_CUDA = 3
VSA_ERR_DEVICE_TIMEOUT = 4
VSA_ERR_INTERNAL = 5
STATIC_WORKSPACE_BYTES = 64 * 1024 * 1024  # VSA_STATIC_WORKSPACE_BYTES in include/vsa.h


class VsaError(RuntimeError):
    def __init__(self, status: int, what: str):
        self.status = status
        super().__init__(f"{what}: {vsa_status_string(status)} (status {status})")


class vsa_shape_t(ctypes.Structure):
    _fields_ = [
        ("batch", ctypes.c_int32),
        ("num_heads", ctypes.c_int32),
        ("head_dim", ctypes.c_int32),
        ("len_text", ctypes.c_int64),
        ("len_audio", ctypes.c_int64),
        ("len_video", ctypes.c_int64),
        ("keep_fraction", ctypes.c_double),
    ]


class vsa_preprocess_args_t(ctypes.Structure):
    _fields_ = [
        ("q_in", ctypes.c_void_p),
        ("k_in", ctypes.c_void_p),
        ("v_in", ctypes.c_void_p),
        ("gate_in", ctypes.c_void_p),
        ("rows_in", ctypes.c_int64),
        ("row_stride", ctypes.c_int64),
        ("src_row", ctypes.c_void_p),
        ("q_norm_weight", ctypes.c_void_p),
        ("k_norm_weight", ctypes.c_void_p),
        ("eps", ctypes.c_float),
        ("rope_dim", ctypes.c_int32),
        ("rope_interleaved", ctypes.c_int32),
        ("rope_cos", ctypes.c_void_p),
        ("rope_sin", ctypes.c_void_p),
        ("q_out", ctypes.c_void_p),
        ("k_out", ctypes.c_void_p),
        ("v_out", ctypes.c_void_p),
        ("gate_out", ctypes.c_void_p),
        ("lengths", ctypes.c_void_p),
    ]


class vsa_output_rows_t(ctypes.Structure):
    _fields_ = [
        ("out", ctypes.c_void_p),
        ("out_rows", ctypes.c_int64),
        ("out_row_stride", ctypes.c_int64),
        ("out_row_map", ctypes.c_void_p),
    ]


class vsa_forward_args_t(ctypes.Structure):
    _fields_ = [
        ("q", ctypes.c_void_p),
        ("k", ctypes.c_void_p),
        ("v", ctypes.c_void_p),
        ("gate", ctypes.c_void_p),
        ("out", ctypes.c_void_p),
        ("rows", ctypes.POINTER(vsa_output_rows_t)),
        ("lengths", ctypes.c_void_p),
        ("preprocessed", ctypes.c_int32),
        ("in_row_stride", ctypes.c_int64),
    ]


_lib = None


def load_library(path: str = LIB_PATH):
    """Load libvsa.so (once). Raises if it is missing: build it first."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(path):
        raise RuntimeError(f"{path} is not built; run block_sparse_video_gb300.build.build() "
                           "(or __graft_entry__.build())")
    lib = ctypes.CDLL(path)
    vp, i32, i64, sz = ctypes.c_void_p, ctypes.c_int32, ctypes.c_int64, ctypes.c_size_t
    sig = {
        "vsa_plan_create": (i32, [ctypes.POINTER(vsa_shape_t), ctypes.c_int, ctypes.POINTER(vp)]),
        "vsa_plan_create_subblock": (i32, [ctypes.POINTER(vsa_shape_t), ctypes.c_double, ctypes.c_int,
                                           ctypes.POINTER(vp)]),
        "vsa_plan_info": (i32, [vp, ctypes.POINTER(i64), ctypes.POINTER(i64), ctypes.POINTER(sz)]),
        "vsa_forward": (i32, [vp, vp, vp, vp, vp, vp, vp, sz, vp]),
        "vsa_preprocess": (i32, [vp, ctypes.POINTER(vsa_preprocess_args_t), vp, sz, vp]),
        "vsa_forward_rows": (i32, [vp, vp, vp, vp, vp, ctypes.POINTER(vsa_output_rows_t), i32, vp, sz, vp]),
        "vsa_forward_lengths": (i32, [vp, vp, vp, vp, vp, vp, vp, vp, sz, vp]),
        "vsa_forward_ex": (i32, [vp, ctypes.POINTER(vsa_forward_args_t), vp, sz, vp]),
        "vsa_forward_preprocessed": (i32, [vp, vp, vp, vp, vp, vp, vp, sz, vp]),
        "vsa_plan_host_path_bytes": (i32, [vp, ctypes.POINTER(sz)]),
        "vsa_plan_host_path_group": (i32, [vp, i32, ctypes.POINTER(i32), ctypes.POINTER(i32), ctypes.POINTER(i32),
                                           ctypes.POINTER(sz), ctypes.POINTER(sz), ctypes.POINTER(sz),
                                           ctypes.POINTER(sz)]),
        "vsa_forward_host": (i32, [vp, vp, vp, vp, vp, vp, vp, sz, vp]),
        "vsa_debug_views": (i32, [vp, vp] + [ctypes.POINTER(vp)] * 5),
        "vsa_check": (i32, [vp, vp, vp]),
        "vsa_plan_set_stage_events": (i32, [vp, ctypes.POINTER(vp)]),
        "vsa_forward_static_workspace": (i32, [vp, vp, vp, vp, vp, vp, vp]),
        "vsa_check_static_workspace": (i32, [vp, vp]),
        "vsa_diag_wait_timeout_static": (i32, [vp, ctypes.c_int, vp]),
        "vsa_diag_wait_timeout": (i32, [vp, vp, ctypes.c_int, vp]),
        "vsa_plan_destroy": (None, [vp]),
        "vsa_status_string": (ctypes.c_char_p, [i32]),
    }
    for name, (res, args) in sig.items():
        fn = getattr(lib, name)
        fn.restype = res
        fn.argtypes = args
    _lib = lib
    return lib


def header_functions(path: str = HEADER_PATH):
    """Names of the functions include/vsa.h declares."""
    text = open(path).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(vsa_[a-z_]+)\s*\(", text)))


def vsa_status_string(status: int) -> str:
    return load_library().vsa_status_string(int(status)).decode()


def _check(status: int, what: str):
    if status != VSA_OK:
        raise VsaError(status, what)


def _ptr(t):
    if t is None:
        return None
    return ctypes.c_void_p(t.data_ptr())


def _stream_handle(stream):
    if stream is None:
        stream = torch.cuda.current_stream()
    return ctypes.c_void_p(stream.cuda_stream)


def vsa_plan_create(batch, num_heads, len_text, len_audio, len_video, keep_fraction,
                    head_dim=128, device=0):
    """Returns an opaque plan handle (an int). Host only."""
    shape = vsa_shape_t(batch, num_heads, head_dim, len_text, len_audio, len_video, keep_fraction)
    out = ctypes.c_void_p()
    _check(load_library().vsa_plan_create(ctypes.byref(shape), int(device), ctypes.byref(out)),
           "vsa_plan_create")
    return out.value


def vsa_plan_create_subblock(batch, num_heads, len_text, len_audio, len_video, sparsity, head_dim=128,
                             device=0):
    """Plan whose selection is the SubBlock router (see vsa.h). Host only."""
    shape = vsa_shape_t(batch, num_heads, head_dim, len_text, len_audio, len_video, 1.0)
    out = ctypes.c_void_p()
    _check(load_library().vsa_plan_create_subblock(ctypes.byref(shape), float(sparsity), int(device),
                                                   ctypes.byref(out)), "vsa_plan_create_subblock")
    return out.value


def vsa_plan_info(plan):
    """(n_tiles T, kept tiles k, workspace bytes)."""
    t, k, ws = ctypes.c_int64(), ctypes.c_int64(), ctypes.c_size_t()
    _check(load_library().vsa_plan_info(plan, ctypes.byref(t), ctypes.byref(k), ctypes.byref(ws)),
           "vsa_plan_info")
    return t.value, k.value, ws.value


def vsa_plan_host_path_bytes(plan):
    n = ctypes.c_size_t()
    _check(load_library().vsa_plan_host_path_bytes(plan, ctypes.byref(n)), "vsa_plan_host_path_bytes")
    return n.value


def vsa_plan_host_path_group(plan, group):
    """Layout of one head group of the host path (see vsa.h): a dict with
    n_groups, first_head, heads, offsets (q, k, v, gate, out), tensor_bytes,
    workspace_offset and workspace_bytes. Host only."""
    ng, h0, nh = ctypes.c_int32(), ctypes.c_int32(), ctypes.c_int32()
    offs = (ctypes.c_size_t * 5)()
    tb, wo, wb = ctypes.c_size_t(), ctypes.c_size_t(), ctypes.c_size_t()
    _check(load_library().vsa_plan_host_path_group(plan, int(group), ctypes.byref(ng), ctypes.byref(h0),
                                                   ctypes.byref(nh), offs, ctypes.byref(tb), ctypes.byref(wo),
                                                   ctypes.byref(wb)), "vsa_plan_host_path_group")
    return {"n_groups": ng.value, "first_head": h0.value, "heads": nh.value, "offsets": list(offs),
            "tensor_bytes": tb.value, "workspace_offset": wo.value, "workspace_bytes": wb.value}


def vsa_plan_destroy(plan):
    if plan:
        load_library().vsa_plan_destroy(plan)


def _check_lengths(lengths, device):
    if (lengths.dtype != torch.int64 or lengths.numel() != 3 or not lengths.is_contiguous()
            or lengths.device != device):
        raise ValueError(f"lengths: expected a contiguous int64 [3] tensor on {device}")
    return lengths


def _check_tensor(x, name, shape, device=None):
    if x.dtype != torch.bfloat16 or tuple(x.shape) != tuple(shape) or not x.is_contiguous():
        raise ValueError(f"{name}: expected contiguous bf16 {tuple(shape)}, got {x.dtype} {tuple(x.shape)}")
    if device is not None and x.device != device:
        raise ValueError(f"{name}: expected a tensor on {device}, got {x.device}")


def _check_head_slice(x, name, shape, device):
    """A bf16 [B, N, H, 128] tensor whose token rows may be wider than H x 128
    channels (a head slice of a wider projection). Returns its row stride in
    elements."""
    if (x.dtype != torch.bfloat16 or tuple(x.shape) != tuple(shape) or x.device != device
            or x.stride(3) != 1 or x.stride(2) != 128):
        raise ValueError(f"{name}: expected bf16 {tuple(shape)} on {device} with contiguous heads of 128 channels")
    if shape[0] > 1 and x.stride(0) != shape[1] * x.stride(1):
        raise ValueError(f"{name}: batches must be N * row stride elements apart")
    return x.stride(1)


def vsa_forward(plan, q, k, v, gate, out, workspace, stream=None):
    """Enqueue the forward on ``stream`` (default: torch's current stream).
    ``gate`` may be None for a SubBlock plan."""
    _check(load_library().vsa_forward(plan, _ptr(q), _ptr(k), _ptr(v), _ptr(gate), _ptr(out),
                                      _ptr(workspace), workspace.numel() * workspace.element_size(),
                                      _stream_handle(stream)), "vsa_forward")


def vsa_preprocess(plan, args, workspace, stream=None):
    """Enqueue the fused preprocessing; ``args`` is a filled vsa_preprocess_args_t."""
    _check(load_library().vsa_preprocess(plan, ctypes.byref(args), _ptr(workspace),
                                         workspace.numel() * workspace.element_size(),
                                         _stream_handle(stream)), "vsa_preprocess")


def vsa_forward_preprocessed(plan, q, k, v, gate, out, workspace, stream=None):
    """Enqueue the forward over inputs packed by vsa_preprocess into ``workspace``."""
    _check(load_library().vsa_forward_preprocessed(plan, _ptr(q), _ptr(k), _ptr(v), _ptr(gate), _ptr(out),
                                                   _ptr(workspace),
                                                   workspace.numel() * workspace.element_size(),
                                                   _stream_handle(stream)), "vsa_forward_preprocessed")


def vsa_forward_rows(plan, q, k, v, gate, rows, preprocessed, workspace, stream=None):
    """Enqueue the forward writing its rows through ``rows`` (a vsa_output_rows_t)."""
    _check(load_library().vsa_forward_rows(plan, _ptr(q), _ptr(k), _ptr(v), _ptr(gate), ctypes.byref(rows),
                                           1 if preprocessed else 0, _ptr(workspace),
                                           workspace.numel() * workspace.element_size(),
                                           _stream_handle(stream)), "vsa_forward_rows")


def vsa_forward_lengths(plan, lengths, q, k, v, gate, out, workspace, stream=None):
    """Enqueue the forward of a request whose lengths (int64 [3] on the device:
    text, audio, video) the kernels read at run time; the plan's shape is the
    capacity of the [B, N_cap, H, 128] buffers."""
    _check(load_library().vsa_forward_lengths(plan, _ptr(lengths), _ptr(q), _ptr(k), _ptr(v), _ptr(gate),
                                              _ptr(out), _ptr(workspace),
                                              workspace.numel() * workspace.element_size(),
                                              _stream_handle(stream)), "vsa_forward_lengths")


def vsa_forward_ex(plan, args, workspace, stream=None):
    """Enqueue the general forward; ``args`` is a filled vsa_forward_args_t."""
    _check(load_library().vsa_forward_ex(plan, ctypes.byref(args), _ptr(workspace),
                                         workspace.numel() * workspace.element_size(),
                                         _stream_handle(stream)), "vsa_forward_ex")


def vsa_forward_host(plan, q, k, v, gate, out, device_buffer, stream=None):
    """Forward on host (ideally pinned) tensors; blocks until ``out`` is filled."""
    _check(load_library().vsa_forward_host(plan, _ptr(q), _ptr(k), _ptr(v), _ptr(gate), _ptr(out),
                                           _ptr(device_buffer),
                                           device_buffer.numel() * device_buffer.element_size(),
                                           _stream_handle(stream)), "vsa_forward_host")


def vsa_forward_static_workspace(plan, q, k, v, gate, out, stream=None):
    """Forward that allocates nothing: the scratch is the library's own fixed-size
    device array (VSA_STATIC_WORKSPACE_BYTES). For callers that cannot allocate
    device memory. Calls that overlap on the GPU race on the shared array."""
    status = load_library().vsa_forward_static_workspace(plan, _ptr(q), _ptr(k), _ptr(v), _ptr(gate),
                                                         _ptr(out), _stream_handle(stream))
    if status == VSA_ERR_UNSUPPORTED:
        raise VsaError(status, "vsa_forward_static_workspace: the plan's workspace exceeds "
                               f"{STATIC_WORKSPACE_BYTES} bytes")
    _check(status, "vsa_forward_static_workspace")


def vsa_check_static_workspace(plan, stream=None):
    """vsa_check for the library-owned array of vsa_forward_static_workspace."""
    _check(load_library().vsa_check_static_workspace(plan, _stream_handle(stream)), "vsa_check_static_workspace")


def vsa_diag_wait_timeout_static(plan, n_ctas=1, stream=None):
    """The diagnostic bounded-wait kernel on the library-owned array (see vsa.h)."""
    _check(load_library().vsa_diag_wait_timeout_static(plan, int(n_ctas), _stream_handle(stream)),
           "vsa_diag_wait_timeout_static")


def vsa_diag_wait_timeout(plan, workspace, n_ctas=1, stream=None):
    """Launch the diagnostic kernel whose bounded waits must run out (see vsa.h)."""
    _check(load_library().vsa_diag_wait_timeout(plan, _ptr(workspace), int(n_ctas), _stream_handle(stream)),
           "vsa_diag_wait_timeout")


def vsa_check(plan, workspace, stream=None):
    """Synchronise and raise VsaError if a bounded wait inside a kernel gave up."""
    _check(load_library().vsa_check(plan, _ptr(workspace), _stream_handle(stream)), "vsa_check")


def vsa_plan_set_stage_events(plan, events):
    """events: four torch.cuda.Event (created with enable_timing=True), or None."""
    if events is None:
        _check(load_library().vsa_plan_set_stage_events(plan, None), "vsa_plan_set_stage_events")
        return
    for e in events:
        if not e.cuda_event:  # torch creates the CUDA event on its first record
            e.record()
    arr = (ctypes.c_void_p * 4)(*[ctypes.c_void_p(e.cuda_event) for e in events])
    _check(load_library().vsa_plan_set_stage_events(plan, arr), "vsa_plan_set_stage_events")


def vsa_debug_views(plan, workspace, batch, num_heads):
    """Torch views of the intermediates in ``workspace``: pooled q/k/v and coarse
    (fp32 [B, H, T, 128]) and the tile selection (int32 [B, H, T, k])."""
    ptrs = [ctypes.c_void_p() for _ in range(5)]
    _check(load_library().vsa_debug_views(plan, _ptr(workspace), *[ctypes.byref(p) for p in ptrs]),
           "vsa_debug_views")
    t, k, _ = vsa_plan_info(plan)
    base = workspace.data_ptr()
    flat = workspace.view(torch.uint8)

    def view(ptr, n_elem, dtype, shape):
        off = ptr.value - base
        nbytes = n_elem * torch.tensor([], dtype=dtype).element_size()
        return flat[off:off + nbytes].view(dtype).view(*shape)

    pooled = batch * num_heads * t * 128
    return dict(
        pooled_q=view(ptrs[0], pooled, torch.float32, (batch, num_heads, t, 128)),
        pooled_k=view(ptrs[1], pooled, torch.float32, (batch, num_heads, t, 128)),
        pooled_v=view(ptrs[2], pooled, torch.float32, (batch, num_heads, t, 128)),
        tile_index=view(ptrs[3], batch * num_heads * t * k, torch.int32, (batch, num_heads, t, k)),
        coarse=view(ptrs[4], pooled, torch.float32, (batch, num_heads, t, 128)),
    )


class VSA:
    """Convenience owner of a plan and its workspace on one device."""

    def __init__(self, batch, num_heads, len_text, len_audio, len_video, keep_fraction=0.2,
                 device="cuda"):
        idx = self._setup(batch, num_heads, len_text, len_audio, len_video, device)
        self._finish(vsa_plan_create(batch, num_heads, len_text, len_audio, len_video, keep_fraction,
                                     device=idx))

    def _setup(self, batch, num_heads, len_text, len_audio, len_video, device):
        self.device = torch.device(device)
        if self.device.type != "cuda":
            raise ValueError("the VSA forward runs on a CUDA device only")
        idx = self.device.index if self.device.index is not None else torch.cuda.current_device()
        self.device = torch.device("cuda", idx)
        self.batch, self.num_heads = batch, num_heads
        self.len_text, self.len_audio, self.len_video = len_text, len_audio, len_video
        self.seq = len_text + len_audio + len_video
        return idx

    def _finish(self, plan):
        self.plan = plan
        self.n_tiles, self.k, self.workspace_bytes = vsa_plan_info(self.plan)
        self.workspace = torch.empty(self.workspace_bytes, dtype=torch.uint8, device=self.device)

    @property
    def shape(self):
        return (self.batch, self.seq, self.num_heads, 128)

    def forward(self, q, k, v, gate, out=None, stream=None):
        for name, x in (("q", q), ("k", k), ("v", v), ("gate", gate)):
            _check_tensor(x, name, self.shape, self.device)
        if out is None:
            out = torch.empty(self.shape, dtype=torch.bfloat16, device=self.device)
        _check_tensor(out, "out", self.shape, self.device)
        vsa_forward(self.plan, q, k, v, gate, out, self.workspace, stream)
        return out

    __call__ = forward

    def preprocess(self, q_in, k_in, v_in, gate_in, q_norm_weight, k_norm_weight, rope_cos=None,
                   rope_sin=None, rope_dim=0, rope_interleaved=True, eps=1e-6, src_row=None, out=None,
                   lengths=None, stream=None):
        """Fused preprocessing of projection rows into packed (q, k, v, gate).

        q_in .. gate_in: bf16 [B, rows_in, H, 128] views sharing one row stride
        (e.g. slices of a merged [B, rows_in, 4, H, 128] projection), channels
        contiguous. q/k_norm_weight: fp32 [H, 128]. rope_cos/sin: fp32
        [N, rope_dim / 2]. src_row: int32 [B, N] or None. out: optional tuple
        of four bf16 [B, N, H, 128] tensors. The pooled statistics stay in this
        object's workspace for forward_preprocessed. lengths: optional device
        int64 [3] (text, audio, video) of a request inside this plan's capacity.
        """
        ins = (q_in, k_in, v_in, gate_in)
        b, h = self.batch, self.num_heads
        for name, x in zip(("q_in", "k_in", "v_in", "gate_in"), ins):
            if (x.dtype != torch.bfloat16 or x.dim() != 4 or x.shape[0] != b or x.shape[2] != h
                    or x.shape[3] != 128 or x.stride(3) != 1 or x.stride(2) != 128 or x.device != self.device):
                raise ValueError(f"{name}: expected bf16 [B, rows_in, H, 128] with contiguous heads on {self.device}")
            if x.shape[1:] != q_in.shape[1:] or x.stride()[:2] != q_in.stride()[:2]:
                raise ValueError("the four projections must share shape and strides")
        rows_in, row_stride = q_in.shape[1], q_in.stride(1)
        if b > 1 and q_in.stride(0) != rows_in * row_stride:
            raise ValueError("batches must be rows_in * row_stride elements apart")
        for name, w in (("q_norm_weight", q_norm_weight), ("k_norm_weight", k_norm_weight)):
            if w.dtype != torch.float32 or tuple(w.shape) != (h, 128) or not w.is_contiguous():
                raise ValueError(f"{name}: expected contiguous fp32 [{h}, 128]")
        if rope_dim:
            for name, t in (("rope_cos", rope_cos), ("rope_sin", rope_sin)):
                if (t is None or t.dtype != torch.float32 or tuple(t.shape) != (self.seq, rope_dim // 2)
                        or not t.is_contiguous()):
                    raise ValueError(f"{name}: expected contiguous fp32 [{self.seq}, {rope_dim // 2}]")
        if src_row is not None and (src_row.dtype != torch.int32 or tuple(src_row.shape) != (b, self.seq)
                                    or not src_row.is_contiguous()):
            raise ValueError(f"src_row: expected contiguous int32 [{b}, {self.seq}]")
        if out is None:
            out = tuple(torch.empty(self.shape, dtype=torch.bfloat16, device=self.device) for _ in range(4))
        for name, x in zip(("q", "k", "v", "gate"), out):
            _check_tensor(x, name, self.shape, self.device)
        args = vsa_preprocess_args_t(
            _ptr(q_in), _ptr(k_in), _ptr(v_in), _ptr(gate_in), rows_in, row_stride, _ptr(src_row),
            _ptr(q_norm_weight), _ptr(k_norm_weight), float(eps), int(rope_dim), 1 if rope_interleaved else 0,
            _ptr(rope_cos) if rope_dim else None, _ptr(rope_sin) if rope_dim else None,
            *[_ptr(x) for x in out], _ptr(_check_lengths(lengths, self.device)) if lengths is not None else None)
        vsa_preprocess(self.plan, args, self.workspace, stream)
        return out

    def forward_preprocessed(self, q, k, v, gate, out=None, stream=None):
        """The forward over tensors packed by ``preprocess`` (same workspace, same stream)."""
        for name, x in (("q", q), ("k", k), ("v", v), ("gate", gate)):
            _check_tensor(x, name, self.shape, self.device)
        if out is None:
            out = torch.empty(self.shape, dtype=torch.bfloat16, device=self.device)
        _check_tensor(out, "out", self.shape, self.device)
        vsa_forward_preprocessed(self.plan, q, k, v, gate, out, self.workspace, stream)
        return out

    def forward_ex(self, q, k, v, gate=None, out=None, out_row_map=None, lengths=None, preprocessed=False,
                   stream=None):
        """The general forward (vsa_forward_ex). ``out``: the packed [B, N, H, 128]
        output, or with ``out_row_map`` (or a non-packed ``out``) output rows as in
        forward_rows; ``lengths``: device int64 [3] of a request inside this
        plan's capacity; ``preprocessed``: the inputs come from ``preprocess``.
        q, k, v and gate may be head slices of wider rows (e.g. ``x[:, :, h0:h0 + H]``
        of a projection with more heads); they must share one row stride."""
        strides = {_check_head_slice(x, name, self.shape, self.device)
                   for name, x in (("q", q), ("k", k), ("v", v)) + ((("gate", gate),) if gate is not None else ())}
        if len(strides) != 1:
            raise ValueError("q, k, v and gate must share one row stride")
        row_stride = strides.pop()
        if out is None:
            out = torch.empty(self.shape, dtype=torch.bfloat16, device=self.device)
        rows = None
        if out_row_map is not None or tuple(out.shape) != self.shape or not out.is_contiguous():
            if out.dtype != torch.bfloat16 or out.dim() < 2 or out.shape[0] != self.batch or not out[0, 0].is_contiguous():
                raise ValueError("out: expected bf16 [B, out_rows, ...] with contiguous rows of H x 128 channels")
            if out_row_map is not None and (out_row_map.dtype != torch.int32 or not out_row_map.is_contiguous()
                                            or tuple(out_row_map.shape) != (self.batch, self.seq)):
                raise ValueError(f"out_row_map: expected contiguous int32 [{self.batch}, {self.seq}]")
            rows = vsa_output_rows_t(_ptr(out), out.shape[1], out.stride(1), _ptr(out_row_map))
        args = vsa_forward_args_t(_ptr(q), _ptr(k), _ptr(v), _ptr(gate), _ptr(out),
                                  ctypes.pointer(rows) if rows is not None else None,
                                  _ptr(_check_lengths(lengths, self.device)) if lengths is not None else None,
                                  1 if preprocessed else 0,
                                  0 if row_stride == self.num_heads * 128 else row_stride)
        vsa_forward_ex(self.plan, args, self.workspace, stream)
        return out

    def forward_lengths(self, lengths, q, k, v, gate, out=None, stream=None):
        """Forward of a request whose lengths (device int64 [3]: text, audio,
        video) are read by the kernels: this object's lengths are the capacity,
        and the tensors are [B, N_cap, H, 128] with the request in rows 0 .. N - 1.
        Capture it once in a CUDA graph and replay it for any request that fits.
        ``gate`` may be None for SubBlock routing."""
        for name, x in (("q", q), ("k", k), ("v", v)) + ((("gate", gate),) if gate is not None else ()):
            _check_tensor(x, name, self.shape, self.device)
        if (lengths.dtype != torch.int64 or lengths.numel() != 3 or not lengths.is_contiguous()
                or lengths.device != self.device):
            raise ValueError(f"lengths: expected a contiguous int64 [3] tensor on {self.device}")
        if out is None:
            out = torch.empty(self.shape, dtype=torch.bfloat16, device=self.device)
        _check_tensor(out, "out", self.shape, self.device)
        vsa_forward_lengths(self.plan, lengths, q, k, v, gate, out, self.workspace, stream)
        return out

    def forward_rows(self, q, k, v, gate, out, out_row_map=None, preprocessed=False, stream=None):
        """The forward writing attention token n of batch b to row out_row_map[b, n]
        (or n) of ``out``, a bf16 [B, out_rows, ...] tensor whose rows hold this
        forward's heads as H x 128 contiguous channels at out.stride(1) elements
        apart (e.g. a slice of a wider buffer). Rows no token maps to are left as
        they are. ``preprocessed``: the inputs come from ``preprocess``."""
        for name, x in (("q", q), ("k", k), ("v", v)) + ((("gate", gate),) if gate is not None else ()):
            _check_tensor(x, name, self.shape, self.device)
        if (out.dtype != torch.bfloat16 or out.dim() < 2 or out.shape[0] != self.batch or out.device != self.device
                or out[0, 0].numel() < self.num_heads * 128 or not out[0, 0].is_contiguous()):
            raise ValueError("out: expected bf16 [B, out_rows, ...] with contiguous rows of H x 128 channels")
        if self.batch > 1 and out.stride(0) != out.shape[1] * out.stride(1):
            raise ValueError("out: batches must be out_rows * row stride elements apart")
        if out_row_map is not None and (out_row_map.dtype != torch.int32 or not out_row_map.is_contiguous()
                                        or tuple(out_row_map.shape) != (self.batch, self.seq)):
            raise ValueError(f"out_row_map: expected contiguous int32 [{self.batch}, {self.seq}]")
        rows = vsa_output_rows_t(_ptr(out), out.shape[1], out.stride(1), _ptr(out_row_map))
        vsa_forward_rows(self.plan, q, k, v, gate, rows, preprocessed, self.workspace, stream)
        return out

    def check(self, stream=None):
        vsa_check(self.plan, self.workspace, stream)

    def debug_views(self):
        return vsa_debug_views(self.plan, self.workspace, self.batch, self.num_heads)

    def __del__(self):
        try:
            vsa_plan_destroy(getattr(self, "plan", None))
        except Exception:
            pass


class SubBlock(VSA):
    """Owner of a SubBlock-routed plan (SGLang Diffusion benchmark page, section
    "How SubBlock Sparse Attention Works"):
    video query tiles keep the k video key tiles of highest estimated softmax
    mass; no coarse branch and no gate. ``sparsity`` is the fraction of key
    tiles that may be dropped."""

    def __init__(self, batch, num_heads, len_text, len_audio, len_video, sparsity=0.75, device="cuda"):
        idx = self._setup(batch, num_heads, len_text, len_audio, len_video, device)
        self.sparsity = sparsity
        self._finish(vsa_plan_create_subblock(batch, num_heads, len_text, len_audio, len_video, sparsity,
                                              device=idx))

    def forward(self, q, k, v, gate=None, out=None, stream=None):
        for name, x in (("q", q), ("k", k), ("v", v)):
            _check_tensor(x, name, self.shape, self.device)
        if out is None:
            out = torch.empty(self.shape, dtype=torch.bfloat16, device=self.device)
        _check_tensor(out, "out", self.shape, self.device)
        vsa_forward(self.plan, q, k, v, None, out, self.workspace, stream)
        return out

    __call__ = forward

    def debug_views(self):
        """sub_q, sub_k: fp32 [B, H, 4T, 128] sub-block means; tile_index: int32 [B, H, T, k]."""
        ptrs = [ctypes.c_void_p() for _ in range(5)]
        _check(load_library().vsa_debug_views(self.plan, _ptr(self.workspace), *[ctypes.byref(p) for p in ptrs]),
               "vsa_debug_views")
        flat = self.workspace.view(torch.uint8)
        base = self.workspace.data_ptr()
        b, h, t, k = self.batch, self.num_heads, self.n_tiles, self.k

        def view(ptr, n_elem, dtype, shape):
            off = ptr.value - base
            nbytes = n_elem * torch.tensor([], dtype=dtype).element_size()
            return flat[off:off + nbytes].view(dtype).view(*shape)

        sub = b * h * 4 * t * 128
        return dict(sub_q=view(ptrs[0], sub, torch.float32, (b, h, 4 * t, 128)),
                    sub_k=view(ptrs[1], sub, torch.float32, (b, h, 4 * t, 128)),
                    tile_index=view(ptrs[3], b * h * t * k, torch.int32, (b, h, t, k)))


__all__ = [
    "VSA", "SubBlock", "VsaError", "vsa_plan_create_subblock", "load_library", "header_functions", "vsa_plan_create", "vsa_plan_info",
    "vsa_forward", "vsa_forward_host", "vsa_preprocess", "vsa_forward_preprocessed", "vsa_forward_rows",
    "vsa_output_rows_t", "vsa_forward_lengths", "vsa_forward_ex", "vsa_forward_args_t",
    "vsa_preprocess_args_t", "vsa_plan_host_path_bytes", "vsa_plan_host_path_group", "vsa_debug_views", "vsa_check",
    "vsa_plan_set_stage_events", "vsa_plan_destroy", "vsa_status_string",
    "vsa_forward_static_workspace", "vsa_diag_wait_timeout",
]
