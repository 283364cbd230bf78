"""Python binding of libvdit (frame-window + reference-frame block-sparse attention
for sm_103a). Argument marshalling only: every step runs in the library's CUDA
kernels; torch provides device memory and the current stream.

The library must be built first (``__graft_entry__.build()`` or
``python -m block_sparse_video_frame_gb300._build``). If it is missing, every
call raises: there is no CPU or eager fallback.

    wf = fold_gamma(w, gamma); cs = rope_table(N, D)    # "Layout Is the ABI", Fig. 5
    q, k, v = qkv_prologue(x, wf, cs, H, D)               # RMSNorm + QKV + RoPE -> [B, H, N, D]
    plan = attn_plan(F, T, W, ref, block_size)          # "Deleting the Mask", Fig. 3
    st = key_stats(q, k, scale)                          # "Unchaining the Softmax"
    o, lse = attn_fwd(plan, q, k, v, st, scale)          # fused tcgen05 kernel
"""
from __future__ import annotations

import ctypes
import os
import threading

from . import configs  # noqa: F401  (plain data, importable without the library)

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "_build", "libvdit.so")

VDIT_OK, VDIT_ERR_INVALID, VDIT_ERR_UNSUPPORTED, VDIT_ERR_CUDA, VDIT_ERR_NOMEM, VDIT_ERR_TIMEOUT = range(6)
MODES = {"auto": 0, "online": 1, "static": 2}
EXPORTED = ("vdit_attn_plan", "vdit_plan_rebuild", "vdit_plan_get_info", "vdit_plan_status",
            "vdit_plan_destroy", "vdit_key_stats_workspace_size", "vdit_key_stats",
            "vdit_attn_fwd", "vdit_last_error", "vdit_version", "vdit_key_stats_noalloc",
            "vdit_set_wait_limit_ns", "vdit_key_stats_framed_workspace_size",
            "vdit_key_stats_framed", "vdit_attn_fwd_framed", "vdit_qkv_fold_gamma",
            "vdit_rope_table", "vdit_qkv_workspace_size", "vdit_qkv_prologue", "vdit_qkv_status",
            "vdit_pipeline_create", "vdit_pipeline_run", "vdit_pipeline_destroy",
            "vdit_pipeline_default_groups", "vdit_set_alloc_fail_after",
            "vdit_set_launch_fail_after", "vdit_plan_block_census", "vdit_attn_plan_part",
            "vdit_attn_fwd_tiles128", "vdit_attn_two_pass_workspace_size", "vdit_attn_fwd_two_pass")
PARTS = {"all": 0, "window": 1, "reference": 2}
TILES = {"frame": 0, "128": 1}


class VditError(RuntimeError):
    def __init__(self, status, msg):
        super().__init__(f"libvdit status {status}: {msg}")
        self.status = status


class PlanInfo(ctypes.Structure):
    _fields_ = [("num_frames", ctypes.c_int32), ("tokens_per_frame", ctypes.c_int32),
                ("window_radius", ctypes.c_int32), ("ref_frame", ctypes.c_int32),
                ("block_size", ctypes.c_int32), ("dense", ctypes.c_int32),
                ("num_tokens", ctypes.c_int64), ("n_qblocks", ctypes.c_int32),
                ("nnz", ctypes.c_int64), ("live_pairs", ctypes.c_int64),
                ("n_segments", ctypes.c_int32), ("n_units", ctypes.c_int32),
                ("n_classes", ctypes.c_int32),
                ("d_row_ptr", ctypes.c_void_p), ("d_col_idx", ctypes.c_void_p),
                ("d_frame_runs", ctypes.c_void_p), ("d_segments", ctypes.c_void_p),
                ("d_units", ctypes.c_void_p), ("d_class_off", ctypes.c_void_p),
                ("part", ctypes.c_int32), ("n_gathers", ctypes.c_int32),
                ("d_gathers", ctypes.c_void_p)]


_lock = threading.Lock()
_lib = None
_I64x3 = ctypes.c_int64 * 3


def load_library(path: str = LIB_PATH):
    """Load libvdit.so and declare its C signatures. Raises if it is not built."""
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        if not os.path.exists(path):
            raise RuntimeError(f"libvdit is not built ({path} missing): run "
                               "`python -c 'import __graft_entry__ as g; g.build()'`")
        lib = ctypes.CDLL(path)
        vp, i32, i64, f32 = ctypes.c_void_p, ctypes.c_int32, ctypes.c_int64, ctypes.c_float
        lib.vdit_attn_plan.argtypes = [i32, i32, i32, i32, i32, vp, ctypes.POINTER(vp)]
        lib.vdit_plan_rebuild.argtypes = [vp, vp]
        lib.vdit_plan_get_info.argtypes = [vp, ctypes.POINTER(PlanInfo)]
        lib.vdit_plan_status.argtypes = [vp, vp, ctypes.POINTER(i32)]
        lib.vdit_plan_destroy.argtypes = [vp]
        lib.vdit_plan_destroy.restype = None
        lib.vdit_key_stats_workspace_size.argtypes = [i32, i32, i32, i32]
        lib.vdit_key_stats_workspace_size.restype = ctypes.c_size_t
        lib.vdit_key_stats.argtypes = [vp, vp, i32, i32, i32, i32, _I64x3, _I64x3, f32, f32,
                                       vp, vp, vp, vp, vp, vp, ctypes.c_size_t, vp]
        lib.vdit_attn_fwd.argtypes = [vp, vp, vp, vp, vp, i32, vp, i32, i32, i32, _I64x3, _I64x3,
                                      _I64x3, _I64x3, f32, vp, vp, vp, i32, vp]
        for fn in ("vdit_attn_plan", "vdit_plan_rebuild", "vdit_plan_get_info",
                   "vdit_plan_status", "vdit_key_stats", "vdit_attn_fwd"):
            getattr(lib, fn).restype = ctypes.c_int
        lib.vdit_last_error.restype = ctypes.c_char_p
        lib.vdit_last_error.argtypes = []
        lib.vdit_version.restype = ctypes.c_char_p
        lib.vdit_version.argtypes = []
        lib.vdit_key_stats_framed_workspace_size.argtypes = [vp, i32, i32, i32]
        lib.vdit_key_stats_framed_workspace_size.restype = ctypes.c_size_t
        lib.vdit_key_stats_framed.argtypes = [vp, vp, vp, i32, i32, i32, _I64x3, _I64x3, f32, f32,
                                              vp, vp, vp, vp, vp, ctypes.c_size_t, vp]
        lib.vdit_key_stats_framed.restype = ctypes.c_int
        lib.vdit_attn_fwd_framed.argtypes = [vp, vp, vp, vp, vp, i32, vp, i32, i32, i32, _I64x3,
                                             _I64x3, _I64x3, _I64x3, f32, vp, vp, vp, i32, vp]
        lib.vdit_attn_fwd_framed.restype = ctypes.c_int
        lib.vdit_set_wait_limit_ns.argtypes = [ctypes.c_uint64]
        lib.vdit_set_wait_limit_ns.restype = None
        _I64x2 = ctypes.c_int64 * 2
        lib.vdit_qkv_fold_gamma.argtypes = [vp, vp, vp, i64, i32, vp]
        lib.vdit_rope_table.argtypes = [vp, i32, i32, ctypes.c_double, vp]
        lib.vdit_qkv_workspace_size.argtypes = [i32, i32]
        lib.vdit_qkv_workspace_size.restype = ctypes.c_size_t
        lib.vdit_qkv_prologue.argtypes = [vp, _I64x2, vp, vp, vp, vp, vp, _I64x3, _I64x3, _I64x3,
                                          i32, i32, i32, i32, i32, f32, vp, ctypes.c_size_t, vp]
        lib.vdit_qkv_status.argtypes = [vp, vp, ctypes.POINTER(i32)]
        for fn in ("vdit_qkv_fold_gamma", "vdit_rope_table", "vdit_qkv_prologue", "vdit_qkv_status"):
            getattr(lib, fn).restype = ctypes.c_int
        lib.vdit_pipeline_create.argtypes = [vp, i32, i32, i32, i32, vp, ctypes.POINTER(vp)]
        lib.vdit_pipeline_create.restype = ctypes.c_int
        lib.vdit_pipeline_run.argtypes = [vp, vp, vp, vp, vp, vp, _I64x3, f32, f32, i32, vp]
        lib.vdit_pipeline_run.restype = ctypes.c_int
        lib.vdit_pipeline_destroy.argtypes = [vp]
        lib.vdit_pipeline_destroy.restype = None
        lib.vdit_pipeline_default_groups.argtypes = [i32, vp, i32]
        lib.vdit_pipeline_default_groups.restype = i32
        lib.vdit_set_alloc_fail_after.argtypes = [i32]
        lib.vdit_set_alloc_fail_after.restype = None
        lib.vdit_attn_plan_part.argtypes = [i32, i32, i32, i32, i32, i32, vp, ctypes.POINTER(vp)]
        lib.vdit_attn_plan_part.restype = ctypes.c_int
        lib.vdit_attn_fwd_tiles128.argtypes = list(lib.vdit_attn_fwd.argtypes)
        lib.vdit_attn_fwd_tiles128.restype = ctypes.c_int
        lib.vdit_attn_two_pass_workspace_size.argtypes = [i32, i32, i32, i32]
        lib.vdit_attn_two_pass_workspace_size.restype = ctypes.c_size_t
        lib.vdit_attn_fwd_two_pass.argtypes = [vp, vp, vp, vp, vp, vp, i32, vp, i32, i32, i32, _I64x3,
                                               _I64x3, _I64x3, _I64x3, f32, vp, vp, vp, i32, i32, vp,
                                               ctypes.c_size_t, vp]
        lib.vdit_attn_fwd_two_pass.restype = ctypes.c_int
        lib.vdit_plan_block_census.argtypes = [vp, i32, vp, vp]
        lib.vdit_plan_block_census.restype = ctypes.c_int
        lib.vdit_set_launch_fail_after.argtypes = [i32]
        lib.vdit_set_launch_fail_after.restype = None
        _lib = lib
        return lib


def _check(status):
    if status != VDIT_OK:
        raise VditError(status, load_library().vdit_last_error().decode())


def _stream(stream):
    import torch
    if stream is None:
        stream = torch.cuda.current_stream()
    return ctypes.c_void_p(stream.cuda_stream)


def _strides(t):
    return _I64x3(*[int(s) for s in t.stride()[:3]])


def _ptr(t):
    return ctypes.c_void_p(0 if t is None else t.data_ptr())


def _check_bhnd(name, t, D=None):
    import torch
    if not isinstance(t, torch.Tensor) or t.dim() != 4:
        raise ValueError(f"{name} must be a 4-D [B, H, N, D] tensor")
    if not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")
    if t.stride(3) != 1:
        raise ValueError(f"{name} must have a contiguous last dimension")
    if D is not None and t.shape[3] != D:
        raise ValueError(f"{name} head dim {t.shape[3]} != {D}")


class Plan:
    """Owns a vdit_plan (device block schedule + work units)."""

    def __init__(self, F, T, W, ref, block_size, stream=None, part="all"):
        lib = load_library()
        h = ctypes.c_void_p()
        pt = PARTS[part] if isinstance(part, str) else int(part)
        if pt == 0:
            _check(lib.vdit_attn_plan(int(F), int(T), int(W), int(ref), int(block_size),
                                      _stream(stream), ctypes.byref(h)))
        else:
            _check(lib.vdit_attn_plan_part(int(F), int(T), int(W), int(ref), int(block_size), pt,
                                           _stream(stream), ctypes.byref(h)))
        self._h = h
        self.info = PlanInfo()
        _check(lib.vdit_plan_get_info(h, ctypes.byref(self.info)))

    @property
    def handle(self):
        return self._h

    @property
    def num_tokens(self):
        return int(self.info.num_tokens)

    @property
    def live_pairs(self):
        return int(self.info.live_pairs)

    def rebuild(self, stream=None):
        _check(load_library().vdit_plan_rebuild(self._h, _stream(stream)))

    def status(self, stream=None) -> int:
        code = ctypes.c_int32()
        st = load_library().vdit_plan_status(self._h, _stream(stream), ctypes.byref(code))
        if st not in (VDIT_OK, VDIT_ERR_TIMEOUT):
            _check(st)
        return int(code.value)

    def block_census(self, tile, stream=None):
        """(full, partial, dead) counts of tile x tile blocks over the N x N token
        pairs, computed on the device (vdit_plan_block_census); synchronises."""
        import torch
        counts = torch.empty(3, dtype=torch.int64, device="cuda")
        _check(load_library().vdit_plan_block_census(self._h, int(tile), _ptr(counts), _stream(stream)))
        return tuple(int(x) for x in counts.cpu().tolist())

    def check(self, stream=None):
        """Synchronise the stream and raise VditError(VDIT_ERR_TIMEOUT) when a kernel
        launched with this plan gave up on an expired wait (its output is then
        incomplete); the status word is cleared either way."""
        code = self.status(stream)
        if code != 0:
            raise VditError(VDIT_ERR_TIMEOUT, f"a kernel's bounded wait expired (site code {code}); "
                                              "its output is incomplete")

    def _device_array(self, ptr, n):
        """Copy of n int32 values of plan-owned device memory (zero-copy view via
        __cuda_array_interface__, then clone)."""
        import torch
        if not n:
            return torch.empty(0, dtype=torch.int32, device="cuda")
        view = torch.as_tensor(_DeviceInts(ptr, int(n)), device="cuda")
        return view.clone()

    def row_ptr(self):
        return self._device_array(self.info.d_row_ptr, self.info.n_qblocks + 1)

    def col_idx(self):
        return self._device_array(self.info.d_col_idx, self.info.nnz)

    def frame_runs(self):
        return self._device_array(self.info.d_frame_runs, 4 * self.info.num_frames).view(-1, 4)

    def segments(self):
        return self._device_array(self.info.d_segments, 8 * self.info.n_segments).view(-1, 8)

    def units(self):
        return self._device_array(self.info.d_units, self.info.n_units)

    def class_offsets(self):
        return self._device_array(self.info.d_class_off, self.info.n_classes + 1)

    def gathers(self):
        """Query tiles of the second attention launch, [n_gathers, 32] int32:
        pieces, rows, the union of the pieces' key runs (lo0, hi0, lo1, hi1), 1,
        its key count, then per piece (segment, first row, rows). Gathered tiles
        hold the ragged tails of 2-8 segments; tail tiles (one piece) are the
        tiles of the last tile pairs of a plan without gathered tiles."""
        return self._device_array(self.info.d_gathers, 32 * self.info.n_gathers).view(-1, 32)

    def close(self):
        if getattr(self, "_h", None) and self._h.value:
            load_library().vdit_plan_destroy(self._h)
            self._h = ctypes.c_void_p()

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass


class _DeviceInts:
    """Describes plan-owned int32 device memory to torch (no copy, no ownership)."""

    def __init__(self, ptr, n):
        self.__cuda_array_interface__ = {"shape": (n,), "typestr": "<i4",
                                         "data": (int(ptr), False), "version": 3,
                                         "strides": None}


def attn_plan(F, T, W, ref, block_size, stream=None, part="all") -> Plan:
    """Block schedule of the frame-window + reference-frame mask (vdit_attn_plan),
    or of one part of it: "window" or "reference" (vdit_attn_plan_part)."""
    return Plan(F, T, W, ref, block_size, stream, part)


def key_stats(q, k, scale, tau=64.0, stream=None, workspace=None, out=None):
    """Per-head key mean, max centred key norm, max query norm, gap bound G and
    eligibility G <= tau (vdit_key_stats). Returns a dict of CUDA tensors
    (written into `out` when given, e.g. the dict a previous call returned)."""
    import torch
    _check_bhnd("q", q)
    _check_bhnd("k", k, q.shape[3])
    if q.dtype != torch.bfloat16 or k.dtype != torch.bfloat16:
        raise ValueError("q and k must be bf16")
    if q.shape != k.shape:
        raise ValueError("q and k must have the same shape")
    B, H, N, D = q.shape
    lib = load_library()
    dev = q.device
    if out is None:
        out = dict(k_mean=torch.empty((B, H, D), dtype=torch.float32, device=dev),
                   k_rmax=torch.empty((B, H), dtype=torch.float32, device=dev),
                   q_nmax=torch.empty((B, H), dtype=torch.float32, device=dev),
                   gap=torch.empty((B, H), dtype=torch.float32, device=dev),
                   eligible=torch.empty((B, H), dtype=torch.uint8, device=dev))
    for name, shape, dt in (("k_mean", (B, H, D), torch.float32), ("k_rmax", (B, H), torch.float32),
                            ("q_nmax", (B, H), torch.float32), ("gap", (B, H), torch.float32),
                            ("eligible", (B, H), torch.uint8)):
        t = out[name]
        if tuple(t.shape) != shape or t.dtype != dt or not t.is_contiguous() or t.device != dev:
            raise ValueError(f"key_stats out[{name!r}] must be a contiguous {dt} {shape} tensor on {dev}")
    need = key_stats_workspace_bytes(B, H, N, D)
    if workspace is None:
        workspace = torch.empty(max(int(need), 16), dtype=torch.uint8, device=dev)
    _check(lib.vdit_key_stats(_ptr(q), _ptr(k), B, H, N, D, _strides(q), _strides(k),
                              float(scale), float(tau), _ptr(out["k_mean"]), _ptr(out["k_rmax"]),
                              _ptr(out["q_nmax"]), _ptr(out["gap"]), _ptr(out["eligible"]),
                              _ptr(workspace), workspace.numel() * workspace.element_size(),
                              _stream(stream)))
    return out


def key_stats_framed(plan: Plan, q, k, scale, tau=64.0, stream=None, workspace=None, out=None):
    """Key statistics with the bound tightened per plan segment (vdit_key_stats_framed).
    Returns dict(k_mean [B,H,D], seg_rmax, seg_gap [B,H,nseg] fp32, seg_eligible [B,H,nseg] u8)."""
    import torch
    _check_bhnd("q", q)
    _check_bhnd("k", k, q.shape[3])
    if q.dtype != torch.bfloat16 or k.dtype != torch.bfloat16 or q.shape != k.shape:
        raise ValueError("q and k must be bf16 tensors of one shape")
    B, H, N, D = q.shape
    if N != plan.num_tokens:
        raise ValueError(f"sequence length {N} != plan's num_tokens {plan.num_tokens}")
    lib = load_library()
    dev = q.device
    S = int(plan.info.n_segments)
    if out is None:
        out = dict(k_mean=torch.empty((B, H, D), dtype=torch.float32, device=dev),
                   seg_rmax=torch.empty((B, H, S), dtype=torch.float32, device=dev),
                   seg_gap=torch.empty((B, H, S), dtype=torch.float32, device=dev),
                   seg_eligible=torch.empty((B, H, S), dtype=torch.uint8, device=dev))
    need = int(lib.vdit_key_stats_framed_workspace_size(plan.handle, B, H, D))
    if workspace is None:
        workspace = torch.empty(max(need, 16), dtype=torch.uint8, device=dev)
    _check(lib.vdit_key_stats_framed(plan.handle, _ptr(q), _ptr(k), B, H, D, _strides(q), _strides(k),
                                     float(scale), float(tau), _ptr(out["k_mean"]),
                                     _ptr(out["seg_rmax"]), _ptr(out["seg_gap"]),
                                     _ptr(out["seg_eligible"]), _ptr(workspace),
                                     workspace.numel() * workspace.element_size(), _stream(stream)))
    return out


def key_stats_framed_workspace_bytes(plan: Plan, B, H, D) -> int:
    return int(load_library().vdit_key_stats_framed_workspace_size(plan.handle, int(B), int(H), int(D)))


def key_stats_workspace_bytes(B, H, N, D) -> int:
    return int(load_library().vdit_key_stats_workspace_size(int(B), int(H), int(N), int(D)))


def _attn_args(plan, q, k, v, stats, scale, mode, out_dtype, with_lse, out, lse):
    """Validated arguments shared by the attention calls."""
    import torch
    _check_bhnd("q", q)
    D = q.shape[3]
    _check_bhnd("k", k, D)
    _check_bhnd("v", v, D)
    for name, t in (("q", q), ("k", k), ("v", v)):
        if t.dtype != torch.bfloat16:
            raise ValueError(f"{name} must be bf16")
        if t.shape != q.shape:
            raise ValueError(f"{name} shape {tuple(t.shape)} != q shape {tuple(q.shape)}")
    B, H, N, _ = q.shape
    if N != plan.num_tokens:
        raise ValueError(f"sequence length {N} != plan's num_tokens {plan.num_tokens}")
    if scale is None:
        scale = D ** -0.5
    m = MODES[mode] if isinstance(mode, str) else int(mode)
    if out is None:
        out = torch.empty((B, H, N, D), dtype=out_dtype or torch.bfloat16, device=q.device)
    _check_bhnd("out", out, D)
    o_code = {torch.bfloat16: 0, torch.float32: 1}[out.dtype]
    if with_lse and lse is None:
        lse = torch.empty((B, H, N), dtype=torch.float32, device=q.device)
    if lse is not None and not (lse.is_contiguous() and lse.dtype == torch.float32
                                and tuple(lse.shape) == (B, H, N)):
        raise ValueError("lse must be a contiguous fp32 [B, H, N] tensor")
    km = kr = el = None
    framed = stats is not None and "seg_rmax" in stats
    if stats is not None:
        km = stats["k_mean"]
        kr, el = (stats["seg_rmax"], stats["seg_eligible"]) if framed else (stats["k_rmax"], stats["eligible"])
    return dict(B=B, H=H, N=N, D=D, scale=float(scale), m=m, out=out, o_code=o_code, lse=lse,
                km=km, kr=kr, el=el, framed=framed)


def attn_fwd(plan: Plan, q, k, v, stats=None, scale=None, mode="auto", out_dtype=None,
             with_lse=True, out=None, lse=None, stream=None, check=True):
    """Fused block-sparse attention (vdit_attn_fwd). Returns (o, lse or None).

    With check=True (the default) the call synchronises the stream and raises
    VditError(VDIT_ERR_TIMEOUT) if the kernel gave up on an expired wait, so an
    incomplete O is never returned silently. check=False keeps the call
    asynchronous; the caller then checks with plan.check() (or plan.status())
    once the stream has passed the call."""
    a = _attn_args(plan, q, k, v, stats, scale, mode, out_dtype, with_lse, out, lse)
    lib = load_library()
    fn = lib.vdit_attn_fwd_framed if a["framed"] else lib.vdit_attn_fwd
    _check(fn(plan.handle, _ptr(q), _ptr(k), _ptr(v), _ptr(a["out"]), a["o_code"], _ptr(a["lse"]),
              a["B"], a["H"], a["D"], _strides(q), _strides(k), _strides(v), _strides(a["out"]),
              a["scale"], _ptr(a["km"]), _ptr(a["kr"]), _ptr(a["el"]), a["m"], _stream(stream)))
    if check:
        plan.check(stream)
    return a["out"], a["lse"]


def attn_fwd_tiles128(plan: Plan, q, k, v, stats=None, scale=None, mode="auto", out_dtype=None,
                      with_lse=True, out=None, lse=None, stream=None, check=True):
    """The attention with the frame-blind tiling of the design before frame
    alignment ("Deleting the Mask", Fig. 3): 128-multiple tiles over the padded
    sequence, mask predicates on straddling tiles (vdit_attn_fwd_tiles128).
    Same results as attn_fwd; an ablation. Per-head statistics only."""
    a = _attn_args(plan, q, k, v, stats, scale, mode, out_dtype, with_lse, out, lse)
    if a["framed"]:
        raise ValueError("the frame-blind tiling takes the per-head statistics (key_stats)")
    _check(load_library().vdit_attn_fwd_tiles128(
        plan.handle, _ptr(q), _ptr(k), _ptr(v), _ptr(a["out"]), a["o_code"], _ptr(a["lse"]), a["B"],
        a["H"], a["D"], _strides(q), _strides(k), _strides(v), _strides(a["out"]), a["scale"],
        _ptr(a["km"]), _ptr(a["kr"]), _ptr(a["el"]), a["m"], _stream(stream)))
    if check:
        plan.check(stream)
    return a["out"], a["lse"]


def two_pass_workspace_bytes(B, H, N, D) -> int:
    return int(load_library().vdit_attn_two_pass_workspace_size(int(B), int(H), int(N), int(D)))


def attn_fwd_two_pass(plan_window: Plan, plan_reference: Plan, q, k, v, stats=None, scale=None,
                      mode="auto", tiles="frame", out_dtype=None, with_lse=True, out=None, lse=None,
                      workspace=None, stream=None, check=True):
    """The attention as the window pass, the reference-frame pass and a merge of
    their fp32 intermediates (vdit_attn_fwd_two_pass), the design before frame
    alignment ("Deleting the Mask"). plan_window / plan_reference: attn_plan(...,
    part="window" / "reference") of one mask. tiles: "frame" (frame-aligned
    passes) or "128" (frame-blind tiling). Same results as attn_fwd; an ablation."""
    import torch
    a = _attn_args(plan_window, q, k, v, stats, scale, mode, out_dtype, with_lse, out, lse)
    if a["framed"]:
        raise ValueError("the two-pass form takes the per-head statistics (key_stats)")
    need = two_pass_workspace_bytes(a["B"], a["H"], a["N"], a["D"])
    if workspace is None:
        workspace = torch.empty(need, dtype=torch.uint8, device=q.device)
    _check(load_library().vdit_attn_fwd_two_pass(
        plan_window.handle, plan_reference.handle, _ptr(q), _ptr(k), _ptr(v), _ptr(a["out"]),
        a["o_code"], _ptr(a["lse"]), a["B"], a["H"], a["D"], _strides(q), _strides(k), _strides(v),
        _strides(a["out"]), a["scale"], _ptr(a["km"]), _ptr(a["kr"]), _ptr(a["el"]), a["m"],
        TILES[str(tiles)], _ptr(workspace), workspace.numel() * workspace.element_size(),
        _stream(stream)))
    if check:
        plan_window.check(stream)
        plan_reference.check(stream)
    return a["out"], a["lse"]


def fold_gamma(w, gamma, out=None, stream=None):
    """W' = bf16(W * gamma) per input channel, once per weight set ("Layout Is
    the ABI": the RMSNorm gain folded into the projection). w: bf16 [rows, C]
    contiguous CUDA tensor; gamma: [C] (any float dtype, read as fp32)."""
    import torch
    if w.dtype != torch.bfloat16 or w.dim() != 2 or not w.is_cuda or not w.is_contiguous():
        raise ValueError("w must be a contiguous bf16 CUDA tensor [rows, C]")
    g = gamma.to(device=w.device, dtype=torch.float32).contiguous()
    if g.numel() != w.shape[1]:
        raise ValueError("gamma must have C entries")
    if out is None:
        out = torch.empty_like(w)
    _check(load_library().vdit_qkv_fold_gamma(_ptr(w), _ptr(g), _ptr(out), w.shape[0], w.shape[1],
                                              _stream(stream)))
    return out


def rope_table(N, D, base=10000.0, device=None, stream=None):
    """fp32 [D/2, N, 2] table of (cos, sin) of n * base^(-2i/D), built on the GPU in fp64."""
    import torch
    t = torch.empty((D // 2, N, 2), dtype=torch.float32, device=device or "cuda")
    _check(load_library().vdit_rope_table(_ptr(t), int(N), int(D), float(base), _stream(stream)))
    return t


def qkv_workspace_bytes(B, N) -> int:
    return int(load_library().vdit_qkv_workspace_size(int(B), int(N)))


def qkv_prologue(x, w_folded, rope, H, D, eps=1e-6, out=None, workspace=None, stream=None):
    """Fused RMSNorm -> q/k/v projection -> rotary embedding -> [B, H, N, D] bf16.
    x: bf16 [B, N, C] CUDA tensor with a contiguous last dimension; w_folded:
    bf16 [3HD, C] from fold_gamma; rope: fp32 [D/2, N, 2] from rope_table (or
    any angle table in that layout). Returns (q, k, v)."""
    import torch
    if x.dtype != torch.bfloat16 or x.dim() != 3 or not x.is_cuda or x.stride(2) != 1:
        raise ValueError("x must be a bf16 CUDA tensor [B, N, C] with a contiguous last dimension")
    B, N, C = x.shape
    if w_folded.shape != (3 * H * D, C) or not w_folded.is_contiguous():
        raise ValueError(f"w_folded must be contiguous [{3 * H * D}, {C}]")
    if rope.shape != (D // 2, N, 2) or rope.dtype != torch.float32 or not rope.is_contiguous():
        raise ValueError(f"rope must be a contiguous fp32 [{D // 2}, {N}, 2] table")
    if out is None:
        out = tuple(torch.empty((B, H, N, D), dtype=torch.bfloat16, device=x.device) for _ in range(3))
    for name, t in zip("qkv", out):
        _check_bhnd(name, t, D)
    need = qkv_workspace_bytes(B, N)
    if workspace is None:
        workspace = torch.zeros(need, dtype=torch.uint8, device=x.device)
    elif workspace.numel() < need:
        raise ValueError(f"workspace needs {need} bytes")
    xs = (ctypes.c_int64 * 2)(int(x.stride(0)), int(x.stride(1)))
    q, k, v = out
    _check(load_library().vdit_qkv_prologue(
        _ptr(x), xs, _ptr(w_folded), _ptr(rope), _ptr(q), _ptr(k), _ptr(v), _strides(q),
        _strides(k), _strides(v), B, N, C, int(H), int(D), float(eps), _ptr(workspace),
        workspace.numel(), _stream(stream)))
    return q, k, v


def qkv_status(workspace, stream=None) -> int:
    """Synchronise, return and clear the status word of a prologue workspace (0 = no expired wait)."""
    code = ctypes.c_int32(0)
    load_library().vdit_qkv_status(_ptr(workspace), _stream(stream), ctypes.byref(code))
    return code.value


class Pipeline:
    """Head-group pipelined attention over HOST tensors ("Hiding the Collective",
    Fig. 2): each group of heads is copied in, gets its key statistics and
    attention, and is copied out, on four streams (copy-in, two compute, copy-out),
    so the middle transfers hide behind other groups' attention (vdit_pipeline_*)."""

    def __init__(self, plan: "Plan", B, H, D, groups):
        """groups: a count (equal split), 0 (the library's tapered schedule) or a
        sequence of per-group head counts."""
        lib = load_library()
        h = ctypes.c_void_p()
        sizes = None
        if not isinstance(groups, int):
            sizes = (ctypes.c_int32 * len(groups))(*[int(g) for g in groups])
            groups = len(groups)
        _check(lib.vdit_pipeline_create(plan.handle, int(B), int(H), int(D), int(groups),
                                        ctypes.cast(sizes, ctypes.c_void_p) if sizes is not None else None,
                                        ctypes.byref(h)))
        self._h = h
        self.plan = plan            # the pipeline keeps using the plan's device schedule
        self.B, self.H, self.D, self.groups = int(B), int(H), int(D), groups
        # host tensors of runs whose copies may still be in flight, each with an
        # event recorded after the run: they stay referenced until it completes
        self._inflight = []

    def run(self, q_h, k_h, v_h, o_h, scale, lse_h=None, tau=64.0, mode="auto", stream=None,
            check=True):
        """q_h, k_h, v_h, o_h: bf16 CPU tensors (pinned for overlap) indexed
        [B, H, N, D] with identical strides and d contiguous; lse_h: optional fp32
        [B, H, N] contiguous CPU tensor. The host tensors stay referenced by the
        pipeline until the run's copies have completed.

        With check=True (the default) the call synchronises the stream, so o_h is
        complete on return, and raises VditError(VDIT_ERR_TIMEOUT) if any of the
        run's attention kernels gave up on an expired wait. check=False keeps the
        run asynchronous: synchronise the stream before reading o_h, and call
        self.plan.check() to learn of expired waits."""
        import torch
        self._inflight = [(ev, held) for ev, held in self._inflight if not ev.query()]
        ts = (q_h, k_h, v_h, o_h)
        for name, t in zip("qkvo", ts):
            if not isinstance(t, torch.Tensor) or t.is_cuda or t.dim() != 4 or t.dtype != torch.bfloat16:
                raise ValueError(f"{name}_h must be a 4-D bf16 CPU tensor")
            if t.stride() != q_h.stride() or t.shape != q_h.shape or t.stride(3) != 1:
                raise ValueError("host tensors must share shape and strides, with d contiguous")
        if tuple(q_h.shape) != (self.B, self.H, self.plan.num_tokens, self.D):
            raise ValueError("host tensors do not match the pipeline's B, H, N, D")
        if lse_h is not None and (lse_h.dtype != torch.float32 or not lse_h.is_contiguous()
                                  or tuple(lse_h.shape) != (self.B, self.H, self.plan.num_tokens)):
            raise ValueError("lse_h must be a contiguous fp32 [B, H, N] CPU tensor")
        status = load_library().vdit_pipeline_run(
            self._h, _ptr(q_h), _ptr(k_h), _ptr(v_h), _ptr(o_h), _ptr(lse_h), _strides(q_h),
            float(scale), float(tau), MODES[mode], _stream(stream))
        # held even when the call failed part-way: copies queued before the error still run
        ev = torch.cuda.Event(enable_timing=False)
        ev.record(stream if stream is not None else torch.cuda.current_stream())
        self._inflight.append((ev, (q_h, k_h, v_h, o_h, lse_h)))
        _check(status)
        if check:
            self.plan.check(stream)
        return o_h

    def close(self):
        if getattr(self, "_h", None) and self._h.value:
            load_library().vdit_pipeline_destroy(self._h)   # waits for the pipeline's streams
            self._h = ctypes.c_void_p()
        self._inflight = []

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass


def default_groups(H: int) -> list:
    """Head counts of the groups that Pipeline(..., groups=0) uses for H heads
    (vdit_pipeline_default_groups; host only)."""
    out = (ctypes.c_int32 * max(1, int(H)))()
    n = load_library().vdit_pipeline_default_groups(int(H), ctypes.cast(out, ctypes.c_void_p), len(out))
    if n <= 0:
        raise ValueError(f"no default schedule for H={H}")
    return [int(out[i]) for i in range(n)]


def set_alloc_fail_after(n: int) -> None:
    """Test hook: the n-th device allocation the library makes from now on fails
    once (VDIT_ERR_NOMEM); n <= 0 switches it off (vdit_set_alloc_fail_after)."""
    load_library().vdit_set_alloc_fail_after(int(n))


def set_launch_fail_after(n: int) -> None:
    """Test hook: the n-th attention launch from now on is refused once, as if
    the launch had failed (VDIT_ERR_CUDA); n <= 0 switches it off
    (vdit_set_launch_fail_after)."""
    load_library().vdit_set_launch_fail_after(int(n))


def set_wait_limit_ns(ns: int) -> None:
    """Bound (ns) of every wait inside attention kernels launched afterwards; 0 = default 1 s."""
    load_library().vdit_set_wait_limit_ns(int(ns))


def version() -> str:
    return load_library().vdit_version().decode()
