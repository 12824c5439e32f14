"""Thin ctypes binding of libmoe.so (the C ABI in include/moe.h).

Argument marshalling only: every step of the forward runs in the library's CUDA kernels.
PyTorch is used for device memory and streams.  Importing this module loads the library
and raises ImportError if it has not been built (``python -m top_routing_grouped_gb300.build``
or ``__graft_entry__.build()``); there is no fallback.
"""
import ctypes
import os

import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libmoe.so")

MOE_OK, MOE_ERR_INVALID_ARG, MOE_ERR_UNSUPPORTED, MOE_ERR_CUDA, MOE_ERR_TIMEOUT, MOE_ERR_INTERNAL = range(6)
MOE_F32, MOE_BF16 = 0, 1
MOE_PATH_AUTO, MOE_PATH_SIMT, MOE_PATH_TC_1SM = 0, 1, 2
_PATHS = {"auto": MOE_PATH_AUTO, "simt": MOE_PATH_SIMT, "tc1": MOE_PATH_TC_1SM}
MOE_FLAG_KEEP_LOGITS, MOE_FLAG_TEST_STALL, MOE_FLAG_RENORM_GATES, MOE_FLAG_TRAINING = 1, 2, 4, 8

if not os.path.exists(LIB_PATH):
    raise ImportError(f"{LIB_PATH} is missing: build it with __graft_entry__.build()")
_lib = ctypes.CDLL(LIB_PATH)


class MoeConfig(ctypes.Structure):
    _fields_ = [("T", ctypes.c_int64), ("d_model", ctypes.c_int32), ("n_experts", ctypes.c_int32),
                ("top_k", ctypes.c_int32), ("d_expert", ctypes.c_int32), ("act_dtype", ctypes.c_int32),
                ("out_dtype", ctypes.c_int32), ("router_temperature", ctypes.c_float),
                ("has_router_bias", ctypes.c_int32), ("path", ctypes.c_int32), ("flags", ctypes.c_uint32),
                ("wait_timeout_ns", ctypes.c_int64)]


class MoeExpertConfig(ctypes.Structure):
    _fields_ = [("max_rows", ctypes.c_int64), ("d_model", ctypes.c_int32), ("n_local_experts", ctypes.c_int32),
                ("n_sources", ctypes.c_int32), ("d_expert", ctypes.c_int32), ("act_dtype", ctypes.c_int32),
                ("path", ctypes.c_int32), ("wait_timeout_ns", ctypes.c_int64)]


class MoeViews(ctypes.Structure):
    _fields_ = [(n, ctypes.c_void_p) for n in (
        "status", "aux", "topk_idx", "topk_gate", "expert_counts", "expert_offsets", "perm_src",
        "perm_slot", "gate_perm", "slot_pos", "logits", "xp", "h", "yp", "expert_psum")]


_P = ctypes.c_void_p
_lib.moe_plan.argtypes = [ctypes.POINTER(MoeConfig), ctypes.POINTER(_P), ctypes.POINTER(ctypes.c_size_t)]
_lib.moe_plan.restype = ctypes.c_int
_lib.moe_plan_destroy.argtypes = [_P]
_lib.moe_plan_destroy.restype = None
_lib.moe_forward.argtypes = [_P] + [_P] * 8 + [ctypes.c_size_t, _P]
_lib.moe_forward.restype = ctypes.c_int
_lib.moe_forward_stage.argtypes = [_P, ctypes.c_int32] + [_P] * 8 + [ctypes.c_size_t, _P]
_lib.moe_forward_stage.restype = ctypes.c_int
_lib.moe_forward_host.argtypes = [_P] + [_P] * 10 + [ctypes.c_size_t, _P]
_lib.moe_forward_host.restype = ctypes.c_int
_lib.moe_stage_count.argtypes = [_P]
_lib.moe_stage_count.restype = ctypes.c_int32
_lib.moe_stage_name.argtypes = [_P, ctypes.c_int32]
_lib.moe_stage_name.restype = ctypes.c_char_p
_lib.moe_aux_loss.argtypes = [_P, _P, _P, _P]
_lib.moe_aux_loss.restype = ctypes.c_int
_lib.moe_workspace_views.argtypes = [_P, _P, ctypes.POINTER(MoeViews)]
_lib.moe_workspace_views.restype = ctypes.c_int
_lib.moe_get_device_status.argtypes = [_P, _P, _P]
_lib.moe_get_device_status.restype = ctypes.c_int
_lib.moe_status_string.argtypes = [ctypes.c_int]
_lib.moe_status_string.restype = ctypes.c_char_p
_lib.moe_backward.argtypes = [_P] * 8 + [ctypes.c_float] + [_P] * 7 + [ctypes.c_size_t, _P]
_lib.moe_backward.restype = ctypes.c_int
_lib.moe_backward_stage.argtypes = [_P, ctypes.c_int32] + [_P] * 7 + [ctypes.c_float] + [_P] * 7 + [ctypes.c_size_t, _P]
_lib.moe_backward_stage.restype = ctypes.c_int
_lib.moe_backward_stage_count.argtypes = [_P]
_lib.moe_backward_stage_count.restype = ctypes.c_int32
_lib.moe_backward_stage_name.argtypes = [_P, ctypes.c_int32]
_lib.moe_backward_stage_name.restype = ctypes.c_char_p
_lib.moe_route_noalloc.argtypes = [_P] * 9 + [_P]
_lib.moe_route_noalloc.restype = ctypes.c_int
_lib.moe_expert_plan.argtypes = [ctypes.POINTER(MoeExpertConfig), ctypes.POINTER(_P), ctypes.POINTER(ctypes.c_size_t)]
_lib.moe_expert_plan.restype = ctypes.c_int
_lib.moe_expert_forward.argtypes = [_P] * 9 + [ctypes.c_size_t, _P]
_lib.moe_expert_forward.restype = ctypes.c_int
_lib.moe_aux_from_totals.argtypes = [ctypes.c_int32, ctypes.c_int32, ctypes.c_int64, _P, _P, _P, _P]
_lib.moe_aux_from_totals.restype = ctypes.c_int
_lib.moe_last_error.argtypes = []
_lib.moe_last_error.restype = ctypes.c_char_p


class MoEError(RuntimeError):
    def __init__(self, status, where):
        self.status = status
        name = _lib.moe_status_string(status).decode()
        detail = _lib.moe_last_error().decode()
        super().__init__(f"{where}: {name}: {detail}")


def _check(status, where):
    if status != MOE_OK:
        raise MoEError(status, where)


def lib():
    return _lib


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream(stream):
    if stream is None:
        stream = torch.cuda.current_stream()
    return ctypes.c_void_p(stream.cuda_stream)


_TORCH = {MOE_F32: torch.float32, MOE_BF16: torch.bfloat16}


class MoEPlan:
    """A plan for one layer shape (names follow the page: T tokens, d = d_model, E experts,
    top-k, F = d_expert, router temperature tau)."""

    def __init__(self, T, d, E, k, F, dtype="bf16", out_dtype=None, tau=1.0, has_bias=False,
                 path="auto", keep_logits=False, test_stall=False, wait_timeout_ns=0, renorm_gates=False,
                 training=False):
        act = MOE_BF16 if dtype == "bf16" else MOE_F32
        out = act if out_dtype is None else (MOE_BF16 if out_dtype == "bf16" else MOE_F32)
        flags = ((MOE_FLAG_KEEP_LOGITS if keep_logits else 0) | (MOE_FLAG_TEST_STALL if test_stall else 0)
                 | (MOE_FLAG_RENORM_GATES if renorm_gates else 0) | (MOE_FLAG_TRAINING if training else 0))
        self.renorm_gates = bool(renorm_gates)
        self.cfg = MoeConfig(int(T), int(d), int(E), int(k), int(F), act, out, float(tau),
                             1 if has_bias else 0, _PATHS[path],
                             flags, int(wait_timeout_ns))
        self.T, self.d, self.E, self.k, self.F = int(T), int(d), int(E), int(k), int(F)
        self.act_dtype, self.out_dtype = _TORCH[act], _TORCH[out]
        self._h = ctypes.c_void_p()
        wsb = ctypes.c_size_t(0)
        _check(_lib.moe_plan(ctypes.byref(self.cfg), ctypes.byref(self._h), ctypes.byref(wsb)), "moe_plan")
        self.workspace_bytes = wsb.value

    @classmethod
    def for_shape(cls, shape, **kw):
        kw.setdefault("renorm_gates", shape.renorm)
        return cls(shape.T, shape.d, shape.E, shape.k, shape.F, dtype=shape.dtype, tau=shape.tau,
                   has_bias=shape.zipf_bias, **kw)

    def __del__(self):
        if getattr(self, "_h", None) and self._h.value:
            _lib.moe_plan_destroy(self._h)
            self._h = ctypes.c_void_p()

    @property
    def handle(self):
        return self._h

    def new_workspace(self, device="cuda"):
        return torch.empty(self.workspace_bytes, dtype=torch.uint8, device=device)

    @property
    def stage_names(self):
        return [_lib.moe_stage_name(self._h, i).decode() for i in range(_lib.moe_stage_count(self._h))]

    def forward(self, x, w_router, bias, w1, w3, w2, y, workspace, stream=None):
        _check(_lib.moe_forward(self._h, _ptr(x), _ptr(w_router), _ptr(bias), _ptr(w1), _ptr(w3), _ptr(w2),
                                _ptr(y), _ptr(workspace), workspace.numel(), _stream(stream)), "moe_forward")

    def forward_stage(self, stage, x, w_router, bias, w1, w3, w2, y, workspace, stream=None):
        _check(_lib.moe_forward_stage(self._h, int(stage), _ptr(x), _ptr(w_router), _ptr(bias), _ptr(w1),
                                      _ptr(w3), _ptr(w2), _ptr(y), _ptr(workspace), workspace.numel(),
                                      _stream(stream)), "moe_forward_stage")

    def forward_host(self, x_host, x_dev, w_router, bias, w1, w3, w2, y_dev, y_host, workspace, stream=None):
        _check(_lib.moe_forward_host(self._h, _ptr(x_host), _ptr(x_dev), _ptr(w_router), _ptr(bias), _ptr(w1),
                                     _ptr(w3), _ptr(w2), _ptr(y_dev), _ptr(y_host), _ptr(workspace),
                                     workspace.numel(), _stream(stream)), "moe_forward_host")

    def backward(self, x, w_router, bias, w1, w3, w2, dy, aux_weight, dx, dw_router, dbias, dw1, dw3, dw2, workspace,
                 stream=None):
        """Gradients of sum(dy * y) + aux_weight * aux into the given fp32 tensors (needs a
        training plan and the workspace of its last forward)."""
        _check(_lib.moe_backward(self._h, _ptr(x), _ptr(w_router), _ptr(bias), _ptr(w1), _ptr(w3), _ptr(w2), _ptr(dy),
                                 float(aux_weight), _ptr(dx), _ptr(dw_router), _ptr(dbias), _ptr(dw1), _ptr(dw3),
                                 _ptr(dw2), _ptr(workspace), workspace.numel(), _stream(stream)), "moe_backward")

    @property
    def backward_stage_names(self):
        return [_lib.moe_backward_stage_name(self._h, i).decode() for i in range(_lib.moe_backward_stage_count(self._h))]

    def backward_stage(self, stage, x, w_router, bias, w1, w3, w2, dy, aux_weight, dx, dw_router, dbias, dw1, dw3, dw2,
                       workspace, stream=None):
        _check(_lib.moe_backward_stage(self._h, int(stage), _ptr(x), _ptr(w_router), _ptr(bias), _ptr(w1), _ptr(w3),
                                       _ptr(w2), _ptr(dy), float(aux_weight), _ptr(dx), _ptr(dw_router), _ptr(dbias),
                                       _ptr(dw1), _ptr(dw3), _ptr(dw2), _ptr(workspace), workspace.numel(),
                                       _stream(stream)), "moe_backward_stage")

    def aux_loss(self, workspace, out=None, stream=None):
        if out is None:
            out = torch.empty((), dtype=torch.float32, device=workspace.device)
        _check(_lib.moe_aux_loss(self._h, _ptr(workspace), _ptr(out), _stream(stream)), "moe_aux_loss")
        return out

    def route_noalloc(self, x, w_router, bias, topk_idx, topk_gate, expert_counts, aux, device_status, stream=None):
        """Routing only, with the library's static scratch (moe_route_noalloc): for callers
        that cannot allocate device memory.  All outputs are caller-provided tensors;
        device_status (one int32/uint32 element) receives 0 or the error a kernel recorded."""
        _check(_lib.moe_route_noalloc(self._h, _ptr(x), _ptr(w_router), _ptr(bias), _ptr(topk_idx),
                                      _ptr(topk_gate), _ptr(expert_counts), _ptr(aux), _ptr(device_status),
                                      _stream(stream)),
               "moe_route_noalloc")

    def device_status(self, workspace, stream=None):
        """Synchronises the stream; returns the status code (MOE_OK == 0)."""
        return _lib.moe_get_device_status(self._h, _ptr(workspace), _stream(stream))

    def views(self, workspace):
        """Tensors viewing the workspace's intermediates of the last forward."""
        v = MoeViews()
        _check(_lib.moe_workspace_views(self._h, _ptr(workspace), ctypes.byref(v)), "moe_workspace_views")
        base = workspace.data_ptr()
        N = self.T * self.k

        def view(addr, dtype, shape):
            if not addr:
                return None
            n = 1
            for s in shape:
                n *= s
            off = addr - base
            nbytes = n * torch.empty((), dtype=dtype).element_size()
            return workspace[off:off + nbytes].view(dtype).view(*shape)

        i32, f32, act = torch.int32, torch.float32, self.act_dtype
        return dict(
            status=view(v.status, i32, (8,)), aux=view(v.aux, f32, (1,)),
            topk_idx=view(v.topk_idx, i32, (self.T, self.k)), topk_gate=view(v.topk_gate, f32, (self.T, self.k)),
            expert_counts=view(v.expert_counts, i32, (self.E,)),
            expert_offsets=view(v.expert_offsets, i32, (self.E + 1,)),
            perm_src=view(v.perm_src, i32, (N,)), perm_slot=view(v.perm_slot, i32, (N,)),
            gate_perm=view(v.gate_perm, f32, (N,)), slot_pos=view(v.slot_pos, i32, (N,)),
            logits=view(v.logits, f32, (self.T, self.E)), xp=view(v.xp, act, (N, self.d)),
            h=view(v.h, act, (N, self.F)), yp=view(v.yp, act, (N, self.d)),
            expert_psum=view(v.expert_psum, f32, (self.E,)))


class ExpertPlan:
    """The expert stage of expert parallelism (moe_expert_plan / moe_expert_forward): the
    local experts (E_l of them) on rows received from W sources, W * E_l segments in
    source-major order, at most max_rows rows."""

    def __init__(self, max_rows, d, E_local, n_sources, F, dtype="bf16", path="auto", wait_timeout_ns=0):
        act = MOE_BF16 if dtype == "bf16" else MOE_F32
        self.cfg = MoeExpertConfig(int(max_rows), int(d), int(E_local), int(n_sources), int(F), act, _PATHS[path],
                                   int(wait_timeout_ns))
        self.max_rows, self.d, self.E_local, self.n_sources, self.F = int(max_rows), int(d), int(E_local), \
            int(n_sources), int(F)
        self.act_dtype = _TORCH[act]
        self._h = ctypes.c_void_p()
        wsb = ctypes.c_size_t(0)
        _check(_lib.moe_expert_plan(ctypes.byref(self.cfg), ctypes.byref(self._h), ctypes.byref(wsb)),
               "moe_expert_plan")
        self.workspace_bytes = wsb.value

    def __del__(self):
        if getattr(self, "_h", None) and self._h.value:
            _lib.moe_plan_destroy(self._h)
            self._h = ctypes.c_void_p()

    @property
    def handle(self):
        return self._h

    def new_workspace(self, device="cuda"):
        return torch.empty(self.workspace_bytes, dtype=torch.uint8, device=device)

    def forward(self, seg_counts, x_rows, gates, w1, w3, w2, y_rows, workspace, stream=None):
        _check(_lib.moe_expert_forward(self._h, _ptr(seg_counts), _ptr(x_rows), _ptr(gates), _ptr(w1), _ptr(w3),
                                       _ptr(w2), _ptr(y_rows), _ptr(workspace), workspace.numel(), _stream(stream)),
               "moe_expert_forward")

    def device_status(self, workspace, stream=None):
        """Synchronises the stream; returns the status code (MOE_OK == 0)."""
        return _lib.moe_get_device_status(self._h, _ptr(workspace), _stream(stream))


def aux_from_totals(E, k, T, counts, psum, out=None, stream=None):
    """The balancing scalar from per-expert totals (moe_aux_from_totals): counts [E] int32 and
    psum [E] fp32 on the device; returns a device fp32 scalar."""
    if out is None:
        out = torch.empty((), dtype=torch.float32, device=counts.device)
    _check(_lib.moe_aux_from_totals(int(E), int(k), int(T), _ptr(counts), _ptr(psum), _ptr(out), _stream(stream)),
           "moe_aux_from_totals")
    return out
