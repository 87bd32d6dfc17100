"""GB300-native two-stage quantized MoE expert computation.

Python binding of libmoe_gb300.so (include/moe.h): argument marshalling only.
Every step of the forward pass runs in the library's CUDA kernels; PyTorch
supplies device memory and streams. If the library is missing or the GPU is
not a GB300, calls raise -- there is no fallback path.
"""
import ctypes
import os

import torch

from . import build as _build

ACT = {"silu": 0, "situv2": 1}
ADTYPE = {"bf16": 0, "fp8": 1, "fp4": 2}
STATUS = {0: "ok", 1: "invalid argument", 2: "unsupported", 3: "CUDA error", 4: "out of device memory",
          5: "expert id out of range", 6: "device wait timed out"}
DEVERR_BAD_EXPERT, DEVERR_TIMEOUT, DEVERR_OVERFLOW = 1, 2, 4
INJECT_ALLOC_FAIL = 1

_lib = None


class MoEError(RuntimeError):
    def __init__(self, status, msg):
        super().__init__("%s (%d): %s" % (STATUS.get(status, "?"), status, msg))
        self.status = status


class _SortView(ctypes.Structure):
    _fields_ = [("sorted_ids", ctypes.c_void_p), ("block_expert", ctypes.c_void_p),
                ("expert_count", ctypes.c_void_p), ("expert_offset", ctypes.c_void_p),
                ("active_experts", ctypes.c_void_p), ("meta", ctypes.c_void_p),
                ("tile_m", ctypes.c_int32), ("max_rows", ctypes.c_int64), ("max_blocks", ctypes.c_int64)]


class _WorkspaceView(ctypes.Structure):
    _fields_ = [("sort", _SortView), ("act_codes", ctypes.c_void_p), ("act_scales", ctypes.c_void_p),
                ("inter_codes", ctypes.c_void_p), ("inter_scales", ctypes.c_void_p), ("acc32", ctypes.c_void_p),
                ("act_scale_stride", ctypes.c_int32), ("inter_scale_stride", ctypes.c_int32),
                ("inter_scale_layout", ctypes.c_int32), ("act_sorted_codes", ctypes.c_void_p),
                ("act_sorted_scales", ctypes.c_void_p), ("act_sorted_scale_stride", ctypes.c_int32),
                ("a16_terms", ctypes.c_int32)]


def library_path():
    return _build.LIB


def lib():
    """Load libmoe_gb300.so (building it first if needed); raises if that fails."""
    global _lib
    if _lib is None:
        path = _build.LIB
        if not os.path.exists(path) or _build._stale():
            path = _build.build()
        L = ctypes.CDLL(path)
        vp, i32, i64, f32 = ctypes.c_void_p, ctypes.c_int, ctypes.c_int64, ctypes.c_float
        L.moe_create.argtypes = [ctypes.POINTER(vp), i32, i32, i32, i32, i32, i32]
        L.moe_destroy.argtypes = [vp]
        L.moe_sort.argtypes = [vp, vp, i32, i32, ctypes.POINTER(_SortView), vp]
        L.moe_forward.argtypes = [vp, vp, vp, vp, i32, vp, vp, vp, vp, i32, f32, f32, i32, vp, vp]
        L.moe_forward_host.argtypes = [vp, vp, vp, vp, i32, vp, vp, vp, vp, i32, f32, f32, i32, vp, vp]
        L.moe_quantize_activations.argtypes = [vp, i32, i32, i32, vp, vp, vp]
        L.moe_quantize_mxfp4.argtypes = [vp, i64, i32, vp, vp, vp]
        L.moe_route.argtypes = [vp, i32, i32, i32, vp, vp, vp]
        L.moe_selftest_wait.argtypes = [vp, i64, i32, vp]
        L.moe_ep_create.argtypes = [ctypes.POINTER(vp), i32, i32, i32, i32, i32, i32, i32]
        L.moe_ep_destroy.argtypes = [vp]
        L.moe_ep_forward.argtypes = [vp, vp, vp, vp, i32, vp, vp, vp, vp, i32, f32, f32, i32, vp, vp]
        L.moe_ep_counts.argtypes = [vp, ctypes.POINTER(ctypes.c_int32)]
        L.moe_ep_get_error.argtypes = [vp, ctypes.POINTER(ctypes.c_int32)]
        L.moe_prepack_size.argtypes = [vp, ctypes.POINTER(ctypes.c_int64)]
        L.moe_prepack.argtypes = [vp, vp, vp, i32, vp, vp]
        L.moe_debug_inject.argtypes = [i32, i64]
        L.moe_get_workspace.argtypes = [vp, ctypes.POINTER(_WorkspaceView)]
        L.moe_get_error.argtypes = [vp, ctypes.POINTER(ctypes.c_int32)]
        L.moe_set_profiling.argtypes = [vp, i32]
        L.moe_read_profile.argtypes = [vp, ctypes.POINTER(ctypes.c_float), ctypes.POINTER(ctypes.c_char_p),
                                       ctypes.POINTER(ctypes.c_int)]
        L.moe_status_string.restype = ctypes.c_char_p
        L.moe_status_string.argtypes = [i32]
        L.moe_last_error_message.restype = ctypes.c_char_p
        L.moe_last_error_message.argtypes = []
        for name in ("moe_create", "moe_destroy", "moe_sort", "moe_forward", "moe_forward_host",
                     "moe_quantize_activations", "moe_quantize_mxfp4", "moe_route", "moe_get_workspace",
                     "moe_selftest_wait", "moe_debug_inject", "moe_prepack_size", "moe_prepack",
                     "moe_ep_create", "moe_ep_destroy", "moe_ep_forward", "moe_ep_counts", "moe_ep_get_error", "moe_get_error",
                     "moe_set_profiling", "moe_read_profile"):
            getattr(L, name).restype = i32
        _lib = L
    return _lib


def _check(status):
    if status != 0:
        raise MoEError(status, lib().moe_last_error_message().decode())


def _ptr(t):
    return ctypes.c_void_p(t.data_ptr()) if t is not None else None


def _stream(stream):
    if stream is None:
        stream = torch.cuda.current_stream()
    return ctypes.c_void_p(stream.cuda_stream)


def _require(t, dtype, name, device=True):
    if not isinstance(t, torch.Tensor):
        raise TypeError("%s must be a torch.Tensor" % name)
    if t.dtype != dtype:
        raise TypeError("%s must be %s, got %s" % (name, dtype, t.dtype))
    if device and not t.is_cuda:
        raise ValueError("%s must be a CUDA tensor" % name)
    if not t.is_contiguous():
        raise ValueError("%s must be contiguous" % name)


class _DevArray:
    """Wraps a raw device pointer for torch.as_tensor via __cuda_array_interface__."""

    def __init__(self, ptr, shape, typestr):
        self.__cuda_array_interface__ = {"shape": tuple(shape), "typestr": typestr, "data": (ptr, False),
                                         "version": 3, "strides": None}


def _view(ptr, shape, dtype):
    typestr = {torch.int32: "<i4", torch.uint8: "|u1", torch.float32: "<f4"}[dtype]
    if any(s == 0 for s in shape):
        return torch.empty(shape, dtype=dtype, device="cuda")
    return torch.as_tensor(_DevArray(ptr, shape, typestr), device="cuda")


class MoE:
    """One context: fixed (hidden, inter, num_experts, topk), up to max_tokens per call."""

    def __init__(self, hidden, inter, num_experts, topk, max_tokens, device=0):
        self.H, self.I, self.E, self.K, self.max_tokens = hidden, inter, num_experts, topk, max_tokens
        self.device = device
        h = ctypes.c_void_p()
        _check(lib().moe_create(ctypes.byref(h), hidden, inter, num_experts, topk, max_tokens, device))
        self._h = h

    def close(self):
        if getattr(self, "_h", None):
            lib().moe_destroy(self._h)
            self._h = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass

    def sort(self, topk_ids, tile_m, stream=None):
        """Run the expert sort; returns a dict of device tensors (copies) and counts."""
        _require(topk_ids, torch.int32, "topk_ids")
        T = topk_ids.shape[0]
        v = _SortView()
        _check(lib().moe_sort(self._h, _ptr(topk_ids), T, tile_m, ctypes.byref(v), _stream(stream)))
        return self._sort_dict(v, stream)

    def _sort_dict(self, v, stream=None):
        torch.cuda.current_stream().synchronize() if stream is None else stream.synchronize()
        meta = _view(v.meta, (4,), torch.int32).cpu()
        nb, na, nr = int(meta[0]), int(meta[1]), int(meta[2])
        return dict(sorted_ids=_view(v.sorted_ids, (nr,), torch.int32).clone(),
                    block_expert=_view(v.block_expert, (nb,), torch.int32).clone(),
                    expert_count=_view(v.expert_count, (self.E,), torch.int32).clone(),
                    expert_offset=_view(v.expert_offset, (self.E + 1,), torch.int32).clone(),
                    active_experts=_view(v.active_experts, (na,), torch.int32).clone(),
                    num_blocks=nb, num_active=na, num_rows=nr, tile_m=v.tile_m)

    def forward(self, x, topk_ids, topk_weights, w13, w13_scale, w2, w2_scale, act="situv2", beta=4.0,
                linear_beta=25.0, a_dtype="bf16", out=None, stream=None):
        """The two-stage forward pass on device tensors; returns out (bf16 [T,H])."""
        _require(x, torch.bfloat16, "x")
        _require(topk_ids, torch.int32, "topk_ids")
        _require(topk_weights, torch.float32, "topk_weights")
        for t, n in ((w13, "w13"), (w13_scale, "w13_scale"), (w2, "w2"), (w2_scale, "w2_scale")):
            _require(t, torch.uint8, n)
        T = x.shape[0]
        if out is None:
            out = torch.empty((T, self.H), dtype=torch.bfloat16, device=x.device)
        _require(out, torch.bfloat16, "out")
        _check(lib().moe_forward(self._h, _ptr(x), _ptr(topk_ids), _ptr(topk_weights), T, _ptr(w13),
                                 _ptr(w13_scale), _ptr(w2), _ptr(w2_scale), ACT[act], float(beta),
                                 float(linear_beta), ADTYPE[a_dtype], _ptr(out), _stream(stream)))
        return out

    def forward_host(self, x, topk_ids, topk_weights, w13, w13_scale, w2, w2_scale, act="situv2", beta=4.0,
                     linear_beta=25.0, a_dtype="bf16", out=None, stream=None):
        """Same, with x / ids / weights / out in (preferably pinned) host memory."""
        _require(x, torch.bfloat16, "x", device=False)
        _require(topk_ids, torch.int32, "topk_ids", device=False)
        _require(topk_weights, torch.float32, "topk_weights", device=False)
        T = x.shape[0]
        if out is None:
            out = torch.empty((T, self.H), dtype=torch.bfloat16, pin_memory=True)
        _check(lib().moe_forward_host(self._h, _ptr(x), _ptr(topk_ids), _ptr(topk_weights), T, _ptr(w13),
                                      _ptr(w13_scale), _ptr(w2), _ptr(w2_scale), ACT[act], float(beta),
                                      float(linear_beta), ADTYPE[a_dtype], _ptr(out), _stream(stream)))
        return out

    def workspace(self):
        """Raw device pointers of the context's workspace."""
        v = _WorkspaceView()
        _check(lib().moe_get_workspace(self._h, ctypes.byref(v)))
        return v

    def last_sort(self):
        """Sort output of the last forward / sort call (device copies)."""
        return self._sort_dict(self.workspace().sort)

    def intermediate(self, rows, a_dtype):
        """Copies of the stage-1 output rows of the last forward: (codes, scales, fmt).

        fmt 'f16' / 'e4m3' / 'e2m1': codes [rows, I * bytes per element], scales [rows, I/32].
        fmt 'e2m1xN' (bf16 activations on the few-rows path, N code terms): codes [rows, N I/2]
        and scales [rows, N I/32], code term t in bytes [t I/2, (t+1) I/2) and scales
        [t I/32, (t+1) I/32); value = sum of the N terms.
        """
        v = self.workspace()
        return self._sorted_rows(v.inter_codes, v.inter_scales, v.inter_scale_stride, v.inter_scale_layout, rows,
                                 self.I, a_dtype, v.a16_terms)

    def sorted_activations(self, rows, a_dtype):
        """Copies of the stage-1 activation operand rows the last forward wrote (x quantised
        per 32 along H, in sorted order): (codes, scales, fmt) with the conventions of
        intermediate(), H in place of I."""
        v = self.workspace()
        return self._sorted_rows(v.act_sorted_codes, v.act_sorted_scales, v.act_sorted_scale_stride,
                                 v.inter_scale_layout, rows, self.H, a_dtype, v.a16_terms)

    def _sorted_rows(self, codes_p, scales_p, stride, layout, rows, width, a_dtype, terms):
        if layout == 2:  # sub-row r * terms + t holds code term t of row r
            codes = _view(codes_p, (rows, terms * width // 2), torch.uint8).clone()
            scales = _view(scales_p, (rows * terms, stride), torch.uint8)[:, :width // 32]
            return codes, scales.reshape(rows, terms * width // 32).clone(), "e2m1x%d" % terms
        bpe = {"bf16": 2, "fp8": 1, "fp4": 0.5}[a_dtype]
        fmt = {"bf16": "f16", "fp8": "e4m3", "fp4": "e2m1"}[a_dtype]
        codes = _view(codes_p, (rows, int(width * bpe)), torch.uint8).clone()
        if layout == 0:
            scales = _view(scales_p, (rows, stride), torch.uint8)[:, :width // 32].clone()
        else:  # 128-row tiles of 512-byte chunks (tensor-core path)
            nb, nc = rows // 128, width // 128
            raw = _view(scales_p, (nb, nc, 32, 4, 4), torch.uint8)  # [tile, chunk, m%32, m/32, kb%4]
            scales = raw.permute(0, 3, 2, 1, 4).reshape(rows, width // 32).clone()
        return codes, scales, fmt

    def set_profiling(self, enable=True):
        _check(lib().moe_set_profiling(self._h, 1 if enable else 0))

    def read_profile(self):
        """[(name, ms)] of each launch group of the last profiled forward."""
        ms = (ctypes.c_float * 8)()
        names = (ctypes.c_char_p * 8)()
        n = ctypes.c_int(8)
        _check(lib().moe_read_profile(self._h, ms, names, ctypes.byref(n)))
        return [(names[i].decode(), float(ms[i])) for i in range(n.value)]

    def prepack(self, w2, w2_scale, a_dtype="bf16", stream=None):
        """Copy w2 / w2_scale into the few-rows stage-2 block layout for a_dtype and bind the
        copy to this context (used by forward calls with this same w2 and a_dtype). Returns
        the packed tensor, which must be kept alive while bound."""
        _require(w2, torch.uint8, "w2")
        _require(w2_scale, torch.uint8, "w2_scale")
        n = ctypes.c_int64(0)
        _check(lib().moe_prepack_size(self._h, ctypes.byref(n)))
        packed = torch.empty(n.value, dtype=torch.uint8, device=w2.device)
        _check(lib().moe_prepack(self._h, _ptr(w2), _ptr(w2_scale), ADTYPE[a_dtype], _ptr(packed), _stream(stream)))
        self._packed = packed
        return packed

    def unbind_prepacked(self):
        _check(lib().moe_prepack(self._h, None, None, 0, None, None))
        self._packed = None

    def selftest_wait(self, limit_ns, complete, stream=None):
        """Run the bounded-wait self-test kernel (see moe_selftest_wait)."""
        _check(lib().moe_selftest_wait(self._h, int(limit_ns), 1 if complete else 0, _stream(stream)))

    def get_error(self):
        """(status, device flag bits); reading clears the device error word."""
        f = ctypes.c_int32(0)
        st = lib().moe_get_error(self._h, ctypes.byref(f))
        if st not in (0, 5, 6):
            _check(st)
        return st, f.value


def quantize_activations(x, a_dtype, stream=None):
    """bf16 [T,H] -> (codes, e8m0 scales [T,H/32]); codes are e4m3 [T,H] for 'fp8', e2m1 pairs
    [T,H/2] for 'fp4', and for 'bf16' f16 bits [T,H] (as uint8 [T,2H]) with one scale per token
    (repeated in all H/32 bytes of the row)."""
    _require(x, torch.bfloat16, "x")
    T, H = x.shape
    width = {"bf16": 2 * H, "fp8": H, "fp4": H // 2}[a_dtype]
    codes = torch.empty((T, width), dtype=torch.uint8, device=x.device)
    scales = torch.empty((T, H // 32), dtype=torch.uint8, device=x.device)
    _check(lib().moe_quantize_activations(_ptr(x), T, H, ADTYPE[a_dtype], _ptr(codes), _ptr(scales),
                                          _stream(stream)))
    return codes, scales


class MoEEP:
    """Expert parallelism emulated on one GPU: `ranks` ranks of experts_per_rank experts,
    dispatch to receive buffers, per-rank forward, fp8 1x32 combine wire (moe_ep_*)."""

    def __init__(self, hidden, inter, experts_per_rank, ranks, topk, max_tokens, device=0):
        self.H, self.R = hidden, ranks
        h = ctypes.c_void_p()
        _check(lib().moe_ep_create(ctypes.byref(h), hidden, inter, experts_per_rank, ranks, topk, max_tokens, device))
        self._h = h

    def close(self):
        if getattr(self, "_h", None):
            lib().moe_ep_destroy(self._h)
            self._h = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass

    def forward(self, x, topk_ids, topk_weights, w13, w13_scale, w2, w2_scale, act="situv2", beta=4.0,
                linear_beta=25.0, a_dtype="bf16", out=None, stream=None):
        _require(x, torch.bfloat16, "x")
        _require(topk_ids, torch.int32, "topk_ids")
        _require(topk_weights, torch.float32, "topk_weights")
        T = x.shape[0]
        if out is None:
            out = torch.empty((T, self.H), dtype=torch.bfloat16, device=x.device)
        _check(lib().moe_ep_forward(self._h, _ptr(x), _ptr(topk_ids), _ptr(topk_weights), T, _ptr(w13),
                                    _ptr(w13_scale), _ptr(w2), _ptr(w2_scale), ACT[act], float(beta),
                                    float(linear_beta), ADTYPE[a_dtype], _ptr(out), _stream(stream)))
        return out

    def counts(self):
        c = (ctypes.c_int32 * self.R)()
        _check(lib().moe_ep_counts(self._h, c))
        return list(c)

    def get_error(self):
        f = ctypes.c_int32(0)
        st = lib().moe_ep_get_error(self._h, ctypes.byref(f))
        if st not in (0, 5, 6):
            _check(st)
        return st, f.value


def debug_inject_alloc_failure(n):
    """The next context creation fails its n-th workspace allocation (MOE_ERR_OOM); n < 0 disarms."""
    _check(lib().moe_debug_inject(INJECT_ALLOC_FAIL, int(n)))


def route(logits, topk, stream=None):
    """Top-k softmax router on the GPU: logits fp32 [T,E] -> (topk_ids int32 [T,K], topk_weights fp32 [T,K])."""
    _require(logits, torch.float32, "logits")
    T, E = logits.shape
    ids = torch.empty((T, topk), dtype=torch.int32, device=logits.device)
    w = torch.empty((T, topk), dtype=torch.float32, device=logits.device)
    _check(lib().moe_route(_ptr(logits), T, E, topk, _ptr(ids), _ptr(w), _stream(stream)))
    return ids, w


def quantize_mxfp4(w, stream=None):
    """fp32 [..., cols] -> (e2m1 codes [..., cols/2], e8m0 scales [..., cols/32]) on the GPU."""
    _require(w, torch.float32, "w")
    cols = w.shape[-1]
    rows = w.numel() // cols
    codes = torch.empty(w.shape[:-1] + (cols // 2,), dtype=torch.uint8, device=w.device)
    scales = torch.empty(w.shape[:-1] + (cols // 32,), dtype=torch.uint8, device=w.device)
    _check(lib().moe_quantize_mxfp4(_ptr(w), rows, cols, _ptr(codes), _ptr(scales), _stream(stream)))
    return codes, scales
