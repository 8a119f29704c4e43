"""Python binding of the C ABI in include/moe_b300.h (ctypes; marshalling only).

Every function has the name of its C entry point without the `moe_` prefix,
takes CUDA torch tensors, checks their dtype/device/contiguity, passes raw
pointers plus the current torch stream, and raises MoeError on a non-zero
status. All arithmetic runs in the CUDA library; torch only allocates the
output buffers. If the library is missing or fails to load, load() raises:
there is no fallback.
"""

from __future__ import annotations

import ctypes
import os
import threading

import torch

from .workloads import Workload

_LIB_PATH = os.path.join(os.path.dirname(os.path.abspath(__file__)), "lib", "libmoe_b300.so")
_lib = None
_lock = threading.Lock()

MOE_DT_F32, MOE_DT_BF16 = 0, 1
MOE_GATE_SOFTMAX, MOE_GATE_NOISY = 0, 1
STATUS = {0: "MOE_OK", 1: "MOE_ERR_INVALID_ARG", 2: "MOE_ERR_UNSUPPORTED", 3: "MOE_ERR_WORKSPACE",
          4: "MOE_ERR_CUDA", 5: "MOE_ERR_DEVICE_TIMEOUT", 6: "MOE_ERR_DEVICE_INDEX",
          7: "MOE_ERR_STATIC_LIMIT"}
PERMUTE_STATIC_MAX_ASSIGN = 1 << 19   # MOE_PERMUTE_STATIC_MAX_ASSIGN

# every symbol include/moe_b300.h declares
EXPORTS = ["moe_status_string", "moe_version", "moe_route_workspace_size", "moe_route",
           "moe_permute_workspace_size",
           "moe_permute", "moe_permute_static", "moe_expert_ffn_workspace_size", "moe_expert_ffn", "moe_combine",
           "moe_workspace_size", "moe_forward", "moe_forward_profiled", "moe_backward_workspace_size",
           "moe_backward", "moe_backward_profiled", "moe_forward_train", "moe_backward_from_forward",
           "moe_device_status", "moe_debug_wait_timeout"]
BWD_PROFILE_EVENTS = 8   # MOE_BWD_PROFILE_EVENTS
PROFILE_EVENTS = 6   # MOE_PROFILE_EVENTS


class MoeError(RuntimeError):
    def __init__(self, status: int, where: str):
        self.status = status
        super().__init__(f"{where}: {STATUS.get(status, status)}")


MOE_ACT_SWIGLU, MOE_ACT_RELU = 0, 1
MOE_COMBINE_ROWS, MOE_COMBINE_SCATTER_ADD = 0, 1


class MoeConfig(ctypes.Structure):
    _fields_ = [("T", ctypes.c_int64), ("d", ctypes.c_int32), ("n_routed", ctypes.c_int32),
                ("n_shared", ctypes.c_int32), ("top_k", ctypes.c_int32), ("d_ff", ctypes.c_int32),
                ("renormalize", ctypes.c_int32), ("gate", ctypes.c_int32),
                ("act_dtype", ctypes.c_int32), ("capacity", ctypes.c_int32),
                ("expert_act", ctypes.c_int32), ("combine", ctypes.c_int32)]


class RouterStats(ctypes.Structure):
    _fields_ = [("lse", ctypes.c_void_p), ("prob_sum", ctypes.c_void_p), ("gate_sum", ctypes.c_void_p)]


def config(w: Workload, T: int | None = None) -> MoeConfig:
    return MoeConfig(T=w.T if T is None else T, d=w.d, n_routed=w.n_routed, n_shared=w.n_shared,
                     top_k=w.top_k, d_ff=w.d_ff, renormalize=int(w.renormalize or w.noisy),
                     gate=MOE_GATE_NOISY if w.noisy else MOE_GATE_SOFTMAX,
                     act_dtype=MOE_DT_F32 if w.fp32 else MOE_DT_BF16, capacity=w.capacity,
                     expert_act=MOE_ACT_RELU if w.act == "relu" else MOE_ACT_SWIGLU,
                     combine=MOE_COMBINE_SCATTER_ADD if w.combine == "scatter" else MOE_COMBINE_ROWS)


def load(path: str = _LIB_PATH) -> ctypes.CDLL:
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        if not os.path.exists(path):
            raise RuntimeError(f"CUDA library not built: {path} (run python -m "
                               "mixture_experts_layer_91_b300.build)")
        lib = ctypes.CDLL(path)
        P, I32, I64, SZ = ctypes.c_void_p, ctypes.c_int32, ctypes.c_int64, ctypes.c_size_t
        C = ctypes.POINTER(MoeConfig)
        sig = {
            "moe_status_string": (ctypes.c_char_p, [ctypes.c_int]),
            "moe_version": (ctypes.c_int, []),
            "moe_route_workspace_size": (SZ, [C]),
            "moe_route": (I32, [C, P, P, P, P, P, P, P, P, P, P, SZ, P]),
            "moe_permute_workspace_size": (SZ, [C]),
            "moe_permute": (I32, [C, P, P, P, SZ, P, P, P, P, P, P]),
            "moe_permute_static": (I32, [C, P, P, P, P, P, P, P, P]),
            "moe_expert_ffn_workspace_size": (SZ, [C]),
            "moe_expert_ffn": (I32, [C, P, P, P, P, P, P, P, SZ, P, P]),
            "moe_combine": (I32, [C, P, P, P, P, P]),
            "moe_workspace_size": (SZ, [C]),
            "moe_forward": (I32, [C, P, P, P, P, P, P, P, P, P, SZ, P, P, P, P, P]),
            "moe_forward_profiled": (I32, [C, P, P, P, P, P, P, P, P, P, SZ, P, P, P, P, P,
                                           ctypes.POINTER(P)]),
            "moe_backward_workspace_size": (SZ, [C]),
            "moe_backward": (I32, [C, P, P, P, P, P, P, P, P, P, P, SZ, P, P, P, P, P, P, P]),
            "moe_backward_profiled": (I32, [C, P, P, P, P, P, P, P, P, P, P, SZ, P, P, P, P, P, P, P,
                                            ctypes.POINTER(P)]),
            "moe_forward_train": (I32, [C, P, P, P, P, P, P, P, P, P, SZ, P, P]),
            "moe_backward_from_forward": (I32, [C, P, P, P, P, P, P, P, P, P, P, SZ, P, P, P, P, P, P, P,
                                                ctypes.POINTER(P)]),
            "moe_device_status": (I32, [P, ctypes.POINTER(I32)]),
            "moe_debug_wait_timeout": (I32, [ctypes.c_uint32, P]),
        }
        for name, (res, args) in sig.items():
            fn = getattr(lib, name)
            fn.restype = res
            fn.argtypes = args
        _lib = lib
        return lib


def _check(status: int, where: str):
    if status != 0:
        raise MoeError(status, where)


def _stream(stream) -> int:
    if stream is None:
        return torch.cuda.current_stream().cuda_stream
    return stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream)


def _ptr(t, dtype=None, name="tensor", optional=False):
    if t is None:
        if optional:
            return None
        raise ValueError(f"{name} is required")
    if not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")
    if dtype is not None and t.dtype != dtype:
        raise ValueError(f"{name} must be {dtype}, got {t.dtype}")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    return t.data_ptr()


def act_dtype(cfg: MoeConfig):
    return torch.bfloat16 if cfg.act_dtype == MOE_DT_BF16 else torch.float32


def workspace_size(cfg: MoeConfig) -> int:
    return load().moe_workspace_size(ctypes.byref(cfg))


def route_workspace_size(cfg: MoeConfig) -> int:
    return load().moe_route_workspace_size(ctypes.byref(cfg))


def permute_workspace_size(cfg: MoeConfig) -> int:
    return load().moe_permute_workspace_size(ctypes.byref(cfg))


def expert_ffn_workspace_size(cfg: MoeConfig) -> int:
    return load().moe_expert_ffn_workspace_size(ctypes.byref(cfg))


def _workspace(nbytes: int, device) -> torch.Tensor:
    return torch.empty(max(nbytes, 16), dtype=torch.uint8, device=device)


def route(cfg, x, W_g, W_noise=None, eps=None, bias=None, *, want_logits=False, want_stats=False,
          workspace=None, stream=None):
    """moe_route. Returns (ids, gates), plus logits [T, E] with want_logits,
    plus a dict of router statistics (lse [T], prob_sum [E], gate_sum [E])
    with want_stats. `workspace`: a uint8 device tensor of at least
    route_workspace_size(cfg) bytes (allocated here when None)."""
    lib = load()
    T, k, E = cfg.T, cfg.top_k, cfg.n_routed
    dev = x.device
    ids = torch.empty(T, k, dtype=torch.int32, device=dev)
    w = torch.empty(T, k, dtype=torch.float32, device=dev)
    logits = torch.empty(T, E, dtype=torch.float32, device=dev) if want_logits else None
    stats = stats_c = None
    if want_stats:
        stats = {"lse": torch.empty(T, dtype=torch.float32, device=dev),
                 "prob_sum": torch.empty(E, dtype=torch.float32, device=dev),
                 "gate_sum": torch.empty(E, dtype=torch.float32, device=dev)}
        stats_c = RouterStats(stats["lse"].data_ptr(), stats["prob_sum"].data_ptr(),
                              stats["gate_sum"].data_ptr())
    ws = _workspace(route_workspace_size(cfg), dev) if workspace is None else workspace
    st = lib.moe_route(ctypes.byref(cfg), _ptr(x, act_dtype(cfg), "x"), _ptr(W_g, torch.float32, "W_g"),
                       _ptr(W_noise, torch.float32, "W_noise", True), _ptr(eps, torch.float32, "eps", True),
                       _ptr(bias, torch.float32, "bias", True), ids.data_ptr(), w.data_ptr(),
                       logits.data_ptr() if logits is not None else None,
                       ctypes.byref(stats_c) if stats_c is not None else None, ws.data_ptr(), ws.numel(),
                       _stream(stream))
    _check(st, "moe_route")
    out = (ids, w)
    if want_logits:
        out = out + (logits,)
    if want_stats:
        out = out + (stats,)
    return out


def permute(cfg, x, topk_ids, *, stream=None) -> dict:
    lib = load()
    T, k, E, d = cfg.T, cfg.top_k, cfg.n_routed, cfg.d
    dev = x.device
    ws = _workspace(permute_workspace_size(cfg), dev)
    out = {"counts": torch.empty(E, dtype=torch.int32, device=dev),
           "offsets": torch.empty(E + 1, dtype=torch.int32, device=dev),
           "dest": torch.empty(T, k, dtype=torch.int32, device=dev),
           "perm_src": torch.empty(T * k, dtype=torch.int32, device=dev),
           "x_perm": torch.empty(T * k, d, dtype=act_dtype(cfg), device=dev)}
    st = lib.moe_permute(ctypes.byref(cfg), _ptr(x, act_dtype(cfg), "x"),
                         _ptr(topk_ids, torch.int32, "topk_ids"), ws.data_ptr(), ws.numel(),
                         out["counts"].data_ptr(), out["offsets"].data_ptr(), out["dest"].data_ptr(),
                         out["perm_src"].data_ptr(), out["x_perm"].data_ptr(), _stream(stream))
    _check(st, "moe_permute")
    return out


def permute_static(cfg, x, topk_ids, *, stream=None) -> dict:
    """moe_permute_static: moe_permute with the library's fixed device scratch
    instead of a workspace (no allocation inside the call)."""
    lib = load()
    T, k, E, d = cfg.T, cfg.top_k, cfg.n_routed, cfg.d
    dev = x.device
    out = {"counts": torch.empty(E, dtype=torch.int32, device=dev),
           "offsets": torch.empty(E + 1, dtype=torch.int32, device=dev),
           "dest": torch.empty(T, k, dtype=torch.int32, device=dev),
           "perm_src": torch.empty(T * k, dtype=torch.int32, device=dev),
           "x_perm": torch.empty(T * k, d, dtype=act_dtype(cfg), device=dev)}
    st = lib.moe_permute_static(ctypes.byref(cfg), _ptr(x, act_dtype(cfg), "x"),
                                _ptr(topk_ids, torch.int32, "topk_ids"), out["counts"].data_ptr(),
                                out["offsets"].data_ptr(), out["dest"].data_ptr(),
                                out["perm_src"].data_ptr(), out["x_perm"].data_ptr(), _stream(stream))
    _check(st, "moe_permute_static")
    return out


def expert_ffn(cfg, x, x_perm, offsets, W1, W3, W2, *, stream=None) -> torch.Tensor:
    lib = load()
    T, k, d, K_s = cfg.T, cfg.top_k, cfg.d, cfg.n_shared
    dt = act_dtype(cfg)
    ws = _workspace(expert_ffn_workspace_size(cfg), x.device)
    out = torch.empty(K_s * T + T * k, d, dtype=torch.float32, device=x.device)
    st = lib.moe_expert_ffn(ctypes.byref(cfg), _ptr(x, dt, "x"), _ptr(x_perm, dt, "x_perm"),
                            _ptr(offsets, torch.int32, "offsets"), _ptr(W1, dt, "W1"),
                            _ptr(W3, dt, "W3", cfg.expert_act == MOE_ACT_RELU),
                            _ptr(W2, dt, "W2"), ws.data_ptr(), ws.numel(), out.data_ptr(), _stream(stream))
    _check(st, "moe_expert_ffn")
    return out


def combine(cfg, out_rows, dest, topk_w, *, stream=None) -> torch.Tensor:
    lib = load()
    y = torch.empty(cfg.T, cfg.d, dtype=act_dtype(cfg), device=out_rows.device)
    st = lib.moe_combine(ctypes.byref(cfg), _ptr(out_rows, torch.float32, "out_rows"),
                         _ptr(dest, torch.int32, "dest"), _ptr(topk_w, torch.float32, "topk_w"),
                         y.data_ptr(), _stream(stream))
    _check(st, "moe_combine")
    return y


def forward(cfg, x, W_g, W_noise, eps, bias, W1, W3, W2, *, workspace=None, y=None,
            routing=False, stream=None):
    """The whole layer. With routing=True also returns (topk_ids, topk_w, counts)."""
    lib = load()
    dt = act_dtype(cfg)
    dev = x.device
    if workspace is None:
        workspace = _workspace(workspace_size(cfg), dev)
    if y is None:
        y = torch.empty(cfg.T, cfg.d, dtype=dt, device=dev)
    ids = w = counts = None
    if routing:
        ids = torch.empty(cfg.T, cfg.top_k, dtype=torch.int32, device=dev)
        w = torch.empty(cfg.T, cfg.top_k, dtype=torch.float32, device=dev)
        counts = torch.empty(cfg.n_routed, dtype=torch.int32, device=dev)
    st = lib.moe_forward(ctypes.byref(cfg), _ptr(x, dt, "x"), _ptr(W_g, torch.float32, "W_g"),
                         _ptr(W_noise, torch.float32, "W_noise", True), _ptr(eps, torch.float32, "eps", True),
                         _ptr(bias, torch.float32, "bias", True), _ptr(W1, dt, "W1"),
                         _ptr(W3, dt, "W3", cfg.expert_act == MOE_ACT_RELU),
                         _ptr(W2, dt, "W2"), _ptr(workspace, torch.uint8, "workspace"), workspace.numel(),
                         _ptr(y, dt, "y"), ids.data_ptr() if routing else None,
                         w.data_ptr() if routing else None, counts.data_ptr() if routing else None,
                         _stream(stream))
    _check(st, "moe_forward")
    return (y, ids, w, counts) if routing else y


def forward_profiled(cfg, x, W_g, W_noise, eps, bias, W1, W3, W2, *, workspace, y, events,
                     stream=None):
    """moe_forward that also records the PROFILE_EVENTS torch.cuda.Event objects
    in `events` at its stage boundaries on the stream it runs on."""
    lib = load()
    dt = act_dtype(cfg)
    if len(events) != PROFILE_EVENTS:
        raise ValueError(f"need {PROFILE_EVENTS} events")
    for e in events:          # torch creates the CUDA event on first record
        if e.cuda_event == 0:
            e.record()
    arr = (ctypes.c_void_p * PROFILE_EVENTS)(*[e.cuda_event for e in events])
    st = lib.moe_forward_profiled(ctypes.byref(cfg), _ptr(x, dt, "x"), _ptr(W_g, torch.float32, "W_g"),
                                  _ptr(W_noise, torch.float32, "W_noise", True),
                                  _ptr(eps, torch.float32, "eps", True), _ptr(bias, torch.float32, "bias", True),
                                  _ptr(W1, dt, "W1"), _ptr(W3, dt, "W3", cfg.expert_act == MOE_ACT_RELU),
                                  _ptr(W2, dt, "W2"),
                                  _ptr(workspace, torch.uint8, "workspace"), workspace.numel(),
                                  _ptr(y, dt, "y"), None, None, None, _stream(stream), arr)
    _check(st, "moe_forward_profiled")
    return y


def backward_workspace_size(cfg: MoeConfig) -> int:
    return load().moe_backward_workspace_size(ctypes.byref(cfg))


def forward_train(cfg, x, W_g, W_noise, eps, bias, W1, W3, W2, *, workspace, y=None, stream=None):
    """moe_forward_train: y, with the backward's state left in `workspace`
    (a uint8 tensor of at least backward_workspace_size(cfg) bytes)."""
    lib = load()
    dt = act_dtype(cfg)
    if y is None:
        y = torch.empty(cfg.T, cfg.d, dtype=dt, device=x.device)
    st = lib.moe_forward_train(ctypes.byref(cfg), _ptr(x, dt, "x"), _ptr(W_g, torch.float32, "W_g"),
                               _ptr(W_noise, torch.float32, "W_noise", True), _ptr(eps, torch.float32, "eps", True),
                               _ptr(bias, torch.float32, "bias", True), _ptr(W1, dt, "W1"),
                               _ptr(W3, dt, "W3", cfg.expert_act == MOE_ACT_RELU), _ptr(W2, dt, "W2"),
                               _ptr(workspace, torch.uint8, "workspace"), workspace.numel(), _ptr(y, dt, "y"),
                               _stream(stream))
    _check(st, "moe_forward_train")
    return y


def backward(cfg, x, W_g, W_noise, eps, bias, W1, W3, W2, dy, *, workspace=None, out=None, events=None,
             from_forward=False, stream=None) -> dict:
    """moe_backward: gradients of the layer for upstream gradient dy.
    Returns a dict dx [T, d] (act dtype), dW_g [d, E], dW_noise [d, E] (noisy
    gate, else None), dW1 / dW3 [G, I, d] (dW3 None for ReLU experts) and
    dW2 [G, d, I], all fp32 but dx. `out` (a dict like the result) reuses
    output buffers; `events` (BWD_PROFILE_EVENTS torch.cuda.Event objects)
    calls moe_backward_profiled, which records them at the stage boundaries.
    from_forward=True calls moe_backward_from_forward on a workspace that
    forward_train filled for the same inputs."""
    lib = load()
    if from_forward and workspace is None:
        raise ValueError("from_forward needs the workspace forward_train filled")
    dt = act_dtype(cfg)
    dev = x.device
    G, I, d, E = cfg.n_routed + cfg.n_shared, cfg.d_ff, cfg.d, cfg.n_routed
    noisy = cfg.gate == MOE_GATE_NOISY
    relu = cfg.expert_act == MOE_ACT_RELU
    if workspace is None:
        workspace = _workspace(backward_workspace_size(cfg), dev)
    f32 = torch.float32
    out = out if out is not None else {"dx": torch.empty(cfg.T, d, dtype=dt, device=dev),
           "dW_g": torch.empty(d, E, dtype=f32, device=dev),
           "dW_noise": torch.empty(d, E, dtype=f32, device=dev) if noisy else None,
           "dW1": torch.empty(G, I, d, dtype=f32, device=dev),
           "dW3": None if relu else torch.empty(G, I, d, dtype=f32, device=dev),
           "dW2": torch.empty(G, d, I, dtype=f32, device=dev)}
    args = [ctypes.byref(cfg), _ptr(x, dt, "x"), _ptr(W_g, torch.float32, "W_g"),
            _ptr(W_noise, torch.float32, "W_noise", True), _ptr(eps, torch.float32, "eps", True),
            _ptr(bias, torch.float32, "bias", True), _ptr(W1, dt, "W1"),
            _ptr(W3, dt, "W3", relu), _ptr(W2, dt, "W2"), _ptr(dy, dt, "dy"),
            _ptr(workspace, torch.uint8, "workspace"), workspace.numel(), _ptr(out["dx"], dt, "dx"),
            _ptr(out["dW_g"], f32, "dW_g"), _ptr(out["dW_noise"], f32, "dW_noise", True),
            _ptr(out["dW1"], f32, "dW1"), _ptr(out["dW3"], f32, "dW3", True), _ptr(out["dW2"], f32, "dW2"),
            _stream(stream)]
    if from_forward:
        arr = None
        if events is not None:
            for e in events:
                if e.cuda_event == 0:
                    e.record()
            arr = (ctypes.c_void_p * BWD_PROFILE_EVENTS)(*[e.cuda_event for e in events])
        _check(lib.moe_backward_from_forward(*args, arr), "moe_backward_from_forward")
        return out
    if events is None:
        _check(lib.moe_backward(*args), "moe_backward")
        return out
    if len(events) != BWD_PROFILE_EVENTS:
        raise ValueError(f"need {BWD_PROFILE_EVENTS} events")
    for e in events:          # torch creates the CUDA event on first record
        if e.cuda_event == 0:
            e.record()
    arr = (ctypes.c_void_p * BWD_PROFILE_EVENTS)(*[e.cuda_event for e in events])
    _check(lib.moe_backward_profiled(*args, arr), "moe_backward_profiled")
    return out


def device_status(*, stream=None) -> tuple[int, int]:
    raw = ctypes.c_int32(0)
    st = load().moe_device_status(_stream(stream), ctypes.byref(raw))
    return st, raw.value


def debug_wait_timeout(limit_us: int, *, stream=None):
    _check(load().moe_debug_wait_timeout(limit_us, _stream(stream)), "moe_debug_wait_timeout")


class MoELayer:
    """One layer's weights and workspace resident on a device; calls moe_forward.

    __call__(x, eps) runs on device tensors; forward_host(x_host, eps_host)
    copies the step's inputs from pinned host memory, runs the layer and
    copies y back, all on the current stream; forward_host_stream runs a
    sequence of host batches with the copies overlapping the forwards.
    """

    def __init__(self, w: Workload, inputs: dict, device="cuda"):
        self.w = w
        self.cfg = config(w)
        dev = torch.device(device)
        self.W_g = inputs["W_g"].to(dev)
        self.W_noise = inputs["W_noise"].to(dev) if inputs["W_noise"] is not None else None
        self.bias = inputs["bias"].to(dev) if inputs["bias"] is not None else None
        self.W1 = inputs["W1"].to(dev)
        self.W3 = inputs["W3"].to(dev) if inputs["W3"] is not None else None
        self.W2 = inputs["W2"].to(dev)
        self.workspace = _workspace(workspace_size(self.cfg), dev)
        self.y = torch.empty(w.T, w.d, dtype=act_dtype(self.cfg), device=dev)
        self.device = dev
        self._streams = {}
        self._bufs = {}

    def __call__(self, x, eps=None, y=None):
        return forward(self.cfg, x, self.W_g, self.W_noise, eps, self.bias, self.W1, self.W3, self.W2,
                       workspace=self.workspace, y=self.y if y is None else y)

    def profiled(self, x, events, eps=None):
        return forward_profiled(self.cfg, x, self.W_g, self.W_noise, eps, self.bias, self.W1, self.W3,
                                self.W2, workspace=self.workspace, y=self.y, events=events)

    def forward_host_stream(self, x_hosts, y_hosts, eps_hosts=None, depth: int = 3):
        """Run the layer over a sequence of batches held in pinned host memory.

        Batch i is copied in on an upload stream, computed on the current
        stream and copied back into y_hosts[i] on a download stream, through
        `depth` device buffers for x and y, so the copies of the next and the
        previous batches overlap the forward of batch i (and a copy never
        waits for the buffer of the step just before). Every copy is enqueued
        before this returns; synchronise the current stream (or the returned
        event) to read y_hosts. Returns the CUDA event recorded after the last
        copy-back.
        """
        n = len(x_hosts)
        if len(y_hosts) != n or (eps_hosts is not None and len(eps_hosts) != n):
            raise ValueError("one output (and eps) buffer per input batch")
        if depth < 2:
            raise ValueError("depth >= 2")
        comp = torch.cuda.current_stream(self.device)
        up = self._streams.setdefault("up", torch.cuda.Stream(self.device))
        down = self._streams.setdefault("down", torch.cuda.Stream(self.device))
        if len(self._bufs.get("x", [])) != depth or (eps_hosts is not None and "eps" not in self._bufs):
            self._bufs["x"] = [torch.empty_like(x_hosts[0], device=self.device) for _ in range(depth)]
            self._bufs["y"] = [torch.empty_like(self.y) for _ in range(depth)]
            if eps_hosts is not None:
                self._bufs["eps"] = [torch.empty_like(eps_hosts[0], device=self.device) for _ in range(depth)]
        xb, yb, eb = self._bufs["x"], self._bufs["y"], self._bufs.get("eps")
        uploaded = [torch.cuda.Event() for _ in range(depth)]
        computed = [torch.cuda.Event() for _ in range(depth)]
        downloaded = [torch.cuda.Event() for _ in range(depth)]
        up.wait_stream(comp)      # buffers may still be read by earlier work on `comp`
        down.wait_stream(comp)
        for i in range(n):
            b = i % depth
            with torch.cuda.stream(up):
                if i >= depth:
                    up.wait_event(computed[b])          # forward i-depth has read xb[b]
                xb[b].copy_(x_hosts[i], non_blocking=True)
                if eb is not None:
                    eb[b].copy_(eps_hosts[i], non_blocking=True)
                uploaded[b].record(up)
            comp.wait_event(uploaded[b])
            if i >= depth:
                comp.wait_event(downloaded[b])          # copy-back i-depth has read yb[b]
            self(xb[b], eb[b] if eb is not None else None, y=yb[b])
            computed[b].record(comp)
            with torch.cuda.stream(down):
                down.wait_event(computed[b])
                y_hosts[i].copy_(yb[b], non_blocking=True)
                downloaded[b].record(down)
        comp.wait_stream(down)
        comp.wait_stream(up)
        done = torch.cuda.Event(enable_timing=True)
        done.record(comp)
        return done

    def forward_host(self, x_host, eps_host=None, y_host=None, x_dev=None, eps_dev=None):
        x_dev = x_dev if x_dev is not None else torch.empty_like(x_host, device=self.device)
        x_dev.copy_(x_host, non_blocking=True)
        if eps_host is not None:
            eps_dev = eps_dev if eps_dev is not None else torch.empty_like(eps_host, device=self.device)
            eps_dev.copy_(eps_host, non_blocking=True)
        y = self(x_dev, eps_dev)
        y_host = y_host if y_host is not None else torch.empty(y.shape, dtype=y.dtype, pin_memory=True)
        y_host.copy_(y, non_blocking=True)
        return y_host
