"""Python binding of libmsk.so: the persistent MoE verify-step kernels.

Argument marshalling only: every step of the verify computation runs in the
library's CUDA kernels.  PyTorch supplies device memory and streams.  There
is no CPU fallback: if the compiled library is missing, every call raises.

The entry points carry the C names (``msk_create``, ``msk_load_layer``,
``msk_layer_step``, ``msk_decode_step``, ...); :class:`Model` bundles them for
weights held in torch tensors.
"""

from __future__ import annotations

import ctypes
import os

import torch

HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(HERE, "lib", "libmsk.so")

MSK_OK = 0
STATUS = {0: "ok", 1: "invalid argument", 2: "shape", 3: "alignment", 4: "bad scale",
          5: "unsupported device", 6: "out of memory", 7: "CUDA error", 8: "timeout",
          9: "not loaded"}
MSK_ERR_INVALID_ARG = 1
MSK_ERR_TIMEOUT = 8
MSK_ERR_NOT_LOADED = 9
TIMELINE_SLOTS = 64
PHASES = ["start", "pro_qkv", "attn", "combine", "oproj", "pool", "router", "topk", "gemm1",
          "gemm2", "mcomb", "unpool", "qkv", "end"]


class MskError(RuntimeError):
    def __init__(self, status, where):
        super().__init__(f"{where}: {STATUS.get(status, status)} ({status})")
        self.status = status


class ModelConfig(ctypes.Structure):
    _fields_ = [
        ("n_layers", ctypes.c_int32), ("hidden", ctypes.c_int32), ("n_q_heads", ctypes.c_int32),
        ("n_kv_heads", ctypes.c_int32), ("head_dim", ctypes.c_int32), ("pooled", ctypes.c_int32),
        ("n_experts", ctypes.c_int32), ("top_k", ctypes.c_int32), ("inter", ctypes.c_int32),
        ("verify_tokens", ctypes.c_int32), ("max_seq", ctypes.c_int32),
        ("prefetch_experts", ctypes.c_int32), ("layer_is_global", ctypes.POINTER(ctypes.c_uint8)),
        ("window", ctypes.c_int32), ("rms_eps", ctypes.c_float), ("rope_theta", ctypes.c_float),
        ("wait_budget_ns", ctypes.c_uint64),
    ]


class Bf16Desc(ctypes.Structure):
    _fields_ = [("data", ctypes.c_void_p), ("rows", ctypes.c_int64), ("cols", ctypes.c_int64),
                ("ld_elems", ctypes.c_int64)]


class Nvfp4Desc(ctypes.Structure):
    _fields_ = [("packed", ctypes.c_void_p), ("scales", ctypes.c_void_p),
                ("tensor_scale", ctypes.c_float), ("rows", ctypes.c_int64), ("cols", ctypes.c_int64)]


class LayerWeightsC(ctypes.Structure):
    _fields_ = [("attn_norm", Bf16Desc), ("moe_norm", Bf16Desc), ("w_qkv", Bf16Desc),
                ("w_o", Bf16Desc), ("w_pool", Bf16Desc), ("w_unpool", Bf16Desc),
                ("w_router", Bf16Desc), ("router_bias", ctypes.c_void_p),
                ("w_gate", ctypes.POINTER(Nvfp4Desc)), ("w_up", ctypes.POINTER(Nvfp4Desc)),
                ("w_down", ctypes.POINTER(Nvfp4Desc))]


#: every symbol include/msk.h declares
SYMBOLS = ["msk_create", "msk_load_layer", "msk_layer_step", "msk_decode_step", "msk_layer_step_tree",
           "msk_decode_step_tree", "msk_step_graph_capture", "msk_step_graph_launch", "msk_set_timing",
           "msk_get_timeline", "msk_set_launch_timing", "msk_get_launch_ms", "msk_set_wait_budget",
           "msk_set_fault_injection", "msk_debug_scratch", "msk_debug_dequant", "msk_debug_quantize", "msk_debug_convert",
           "msk_debug_fp4_gemm",
           "msk_attention_noalloc", "msk_get_info", "msk_status_string", "msk_destroy"]

_lib = None


def load_library(path: str = LIB_PATH):
    """Loads libmsk.so (raises if it was not built)."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(path):
        raise RuntimeError(f"libmsk.so not found at {path}: build it first "
                           "(python -m moe_decode_step_persistent_gb300.build)")
    L = ctypes.CDLL(path)
    vp, i32, i64, u64 = ctypes.c_void_p, ctypes.c_int32, ctypes.c_int64, ctypes.c_uint64
    L.msk_create.argtypes = [ctypes.POINTER(ModelConfig), ctypes.POINTER(vp)]
    L.msk_load_layer.argtypes = [vp, i32, ctypes.POINTER(LayerWeightsC), vp]
    L.msk_layer_step.argtypes = [vp, i32, vp, vp, ctypes.POINTER(i32), vp, vp, i32, vp]
    L.msk_decode_step.argtypes = [vp, vp, vp, ctypes.POINTER(i32), vp, vp, vp]
    L.msk_layer_step_tree.argtypes = [vp, i32, vp, vp, i32, ctypes.POINTER(i32), vp, vp, i32, vp]
    L.msk_decode_step_tree.argtypes = [vp, vp, vp, i32, ctypes.POINTER(i32), vp, vp, vp]
    L.msk_step_graph_capture.argtypes = [vp, vp, vp, vp, vp]
    L.msk_step_graph_launch.argtypes = [vp, i32, ctypes.POINTER(i32), vp]
    L.msk_set_timing.argtypes = [vp, i32]
    L.msk_get_timeline.argtypes = [vp, ctypes.POINTER(ctypes.c_uint64), ctypes.c_size_t,
                                   ctypes.POINTER(ctypes.c_size_t), ctypes.POINTER(i32), ctypes.POINTER(i32)]
    L.msk_set_launch_timing.argtypes = [vp, i32]
    L.msk_get_launch_ms.argtypes = [vp, ctypes.POINTER(ctypes.c_float), i32, ctypes.POINTER(i32)]
    L.msk_set_wait_budget.argtypes = [vp, u64]
    L.msk_set_fault_injection.argtypes = [vp, i32, i32]
    L.msk_debug_scratch.argtypes = [vp, i32, vp, ctypes.c_size_t, ctypes.POINTER(ctypes.c_size_t), vp]
    L.msk_debug_dequant.argtypes = [vp, i32, i32, i32, vp, vp]
    L.msk_debug_quantize.argtypes = [vp, i64, i64, vp, vp, vp]
    L.msk_debug_convert.argtypes = [vp, i64, vp, vp, vp]
    L.msk_debug_fp4_gemm.argtypes = [vp, vp, vp, vp, i32, i32, vp, vp]
    L.msk_attention_noalloc.argtypes = [vp, vp, i32, i32, i32, i32, i32, i32, i32, vp, vp]
    L.msk_get_info.argtypes = [vp, ctypes.POINTER(i32), ctypes.POINTER(i64)]
    L.msk_status_string.argtypes = [i32]
    L.msk_status_string.restype = ctypes.c_char_p
    L.msk_destroy.argtypes = [vp]
    L.msk_destroy.restype = None
    for name in SYMBOLS:
        if name not in ("msk_status_string", "msk_destroy"):
            getattr(L, name).restype = i32
    _lib = L
    return L


def _check(status, where):
    if status != MSK_OK:
        raise MskError(status, where)


def _stream(stream=None):
    s = stream if stream is not None else torch.cuda.current_stream()
    return ctypes.c_void_p(s.cuda_stream)


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _positions(positions):
    return (ctypes.c_int32 * len(positions))(*[int(p) for p in positions])


# ----------------------------------------------------------------------------
# thin wrappers, same names as the C ABI
# ----------------------------------------------------------------------------


def msk_create(cfg: ModelConfig) -> ctypes.c_void_p:
    L = load_library()
    h = ctypes.c_void_p()
    _check(L.msk_create(ctypes.byref(cfg), ctypes.byref(h)), "msk_create")
    return h


def msk_load_layer(handle, layer, weights: LayerWeightsC, stream=None):
    _check(load_library().msk_load_layer(handle, layer, ctypes.byref(weights), _stream(stream)), "msk_load_layer")


def msk_layer_step(handle, layer, hidden, kv_cache, positions, prev_routing=None, routing_out=None,
                   run_prologue=False, stream=None):
    return load_library().msk_layer_step(handle, layer, _ptr(hidden), _ptr(kv_cache), _positions(positions),
                                         _ptr(prev_routing), _ptr(routing_out), int(run_prologue), _stream(stream))


def msk_decode_step(handle, hidden, kv_cache, positions, prev_routing=None, routing_out=None, stream=None):
    return load_library().msk_decode_step(handle, _ptr(hidden), _ptr(kv_cache), _positions(positions),
                                          _ptr(prev_routing), _ptr(routing_out), _stream(stream))


def msk_layer_step_tree(handle, layer, hidden, kv_cache, cache_len, parents, prev_routing=None, routing_out=None,
                        run_prologue=False, stream=None):
    return load_library().msk_layer_step_tree(handle, layer, _ptr(hidden), _ptr(kv_cache), int(cache_len),
                                              _positions(parents), _ptr(prev_routing), _ptr(routing_out),
                                              int(run_prologue), _stream(stream))


def msk_decode_step_tree(handle, hidden, kv_cache, cache_len, parents, prev_routing=None, routing_out=None,
                         stream=None):
    return load_library().msk_decode_step_tree(handle, _ptr(hidden), _ptr(kv_cache), int(cache_len),
                                               _positions(parents), _ptr(prev_routing), _ptr(routing_out),
                                               _stream(stream))


def msk_step_graph_capture(handle, hidden, kv_cache, prev_routing=None, routing_out=None):
    return load_library().msk_step_graph_capture(handle, _ptr(hidden), _ptr(kv_cache), _ptr(prev_routing),
                                                 _ptr(routing_out))


def msk_step_graph_launch(handle, cache_len, parents=None, stream=None):
    par = None if parents is None else _positions(parents)
    return load_library().msk_step_graph_launch(handle, int(cache_len), par, _stream(stream))


def msk_debug_dequant(handle, layer, expert, which, out, stream=None):
    _check(load_library().msk_debug_dequant(handle, layer, expert, which, _ptr(out), _stream(stream)),
           "msk_debug_dequant")


def msk_debug_quantize(x, codes, scales, stream=None):
    _check(load_library().msk_debug_quantize(_ptr(x), x.shape[0], x.shape[1], _ptr(codes), _ptr(scales),
                                             _stream(stream)), "msk_debug_quantize")


def msk_debug_convert(x, e2m1, e4m3, stream=None):
    _check(load_library().msk_debug_convert(_ptr(x), x.numel(), _ptr(e2m1), _ptr(e4m3), _stream(stream)),
           "msk_debug_convert")


def msk_debug_fp4_gemm(a_codes, a_scales, b_codes, b_scales, d, stream=None):
    """d[128][16] = A B^T on the tensor cores (block-scaled NVFP4; see
    include/msk.h).  a_codes [128][K/2], a_scales [128][K/16], b_codes
    [n][K/2], b_scales [n][K/16] uint8; d [128][16] fp32.  Returns the status."""
    return load_library().msk_debug_fp4_gemm(_ptr(a_codes), _ptr(a_scales), _ptr(b_codes), _ptr(b_scales),
                                             b_codes.shape[0], a_codes.shape[1] * 2, _ptr(d), _stream(stream))


def msk_attention_noalloc(q, kv_layer, pos0, window, out, stream=None):
    """Standalone split-KV attention that allocates no device memory (its
    scratch is a fixed array inside the library): for callers that cannot
    allocate at the point of the call.  q: [T][Hq][d] bf16; kv_layer:
    [2][Hkv][max_seq][d] bf16; out: [T][Hq*d] bf16.  Returns the status."""
    T, Hq, d = q.shape
    Hkv, max_seq = kv_layer.shape[1], kv_layer.shape[2]
    return load_library().msk_attention_noalloc(_ptr(q), _ptr(kv_layer), T, Hq, Hkv, d, max_seq, int(pos0),
                                                int(window), _ptr(out), _stream(stream))


def msk_destroy(handle):
    load_library().msk_destroy(handle)


# ----------------------------------------------------------------------------
# Model: descriptors from torch tensors
# ----------------------------------------------------------------------------


def _bf16(t):
    t2 = t if t.dim() == 2 else t.reshape(1, -1)
    assert t2.dtype == torch.bfloat16 and t2.is_cuda and t2.stride(1) == 1
    return Bf16Desc(t2.data_ptr(), t2.shape[0], t2.shape[1], t2.stride(0))


def _fp4_array(trip):
    packed, scales, ts = trip
    n = packed.shape[0]
    arr = (Nvfp4Desc * n)()
    tsh = ts.detach().float().cpu().tolist()
    for e in range(n):
        arr[e] = Nvfp4Desc(packed[e].data_ptr(), scales[e].data_ptr(), tsh[e], packed.shape[1],
                           packed.shape[2] * 2)
    return arr


class Model:
    """A loaded model.  ``dims`` is any object with the workload fields
    (hidden, n_q_heads, n_kv_heads, head_dim, pooled, n_experts, top_k,
    inter, tokens, max_seq, windows, rms_eps, rope_theta)."""

    def __init__(self, dims, prefetch_experts=14, wait_budget_ns=0):
        windows = list(dims.windows)
        self.dims = dims
        self.n_layers = len(windows)
        sliding = [w for w in windows if w > 0]
        if len(set(sliding)) > 1:
            raise ValueError("all sliding-window layers share one window size (msk_model_config.window); "
                             f"got {sorted(set(sliding))}")
        self._glob = (ctypes.c_uint8 * self.n_layers)(*[1 if w == 0 else 0 for w in windows])
        cfg = ModelConfig(self.n_layers, dims.hidden, dims.n_q_heads, dims.n_kv_heads, dims.head_dim,
                          dims.pooled, dims.n_experts, dims.top_k, dims.inter, dims.tokens, dims.max_seq,
                          prefetch_experts, self._glob, sliding[0] if sliding else 0, dims.rms_eps,
                          dims.rope_theta, wait_budget_ns)
        self.handle = msk_create(cfg)
        n = ctypes.c_int32()
        b = ctypes.c_int64()
        _check(load_library().msk_get_info(self.handle, ctypes.byref(n), ctypes.byref(b)), "msk_get_info")
        self.n_ctas = n.value

    def load_layer(self, layer, lt, stream=None):
        """lt: msk_synth.LayerTensors on the current CUDA device."""
        gate, up, down = _fp4_array(lt.gate), _fp4_array(lt.up), _fp4_array(lt.down)
        w = LayerWeightsC(_bf16(lt.attn_norm), _bf16(lt.moe_norm), _bf16(lt.w_qkv), _bf16(lt.w_o),
                          _bf16(lt.w_pool), _bf16(lt.w_unpool), _bf16(lt.w_router),
                          lt.router_bias.data_ptr(), gate, up, down)
        msk_load_layer(self.handle, layer, w, stream)

    def device_bytes(self):
        n = ctypes.c_int32()
        b = ctypes.c_int64()
        _check(load_library().msk_get_info(self.handle, ctypes.byref(n), ctypes.byref(b)), "msk_get_info")
        return b.value

    def layer_step(self, layer, hidden, kv_cache, positions, prev_routing=None, routing_out=None,
                   run_prologue=False, stream=None, check=True):
        st = msk_layer_step(self.handle, layer, hidden, kv_cache, positions, prev_routing, routing_out,
                            run_prologue, stream)
        if check:
            _check(st, "msk_layer_step")
        return st

    def decode_step(self, hidden, kv_cache, positions, prev_routing=None, routing_out=None, stream=None,
                    check=True):
        st = msk_decode_step(self.handle, hidden, kv_cache, positions, prev_routing, routing_out, stream)
        if check:
            _check(st, "msk_decode_step")
        return st

    def layer_step_tree(self, layer, hidden, kv_cache, cache_len, parents, prev_routing=None, routing_out=None,
                        run_prologue=False, stream=None, check=True):
        """One launch verifying a tree of candidates (see msk_layer_step_tree)."""
        st = msk_layer_step_tree(self.handle, layer, hidden, kv_cache, cache_len, parents, prev_routing,
                                 routing_out, run_prologue, stream)
        if check:
            _check(st, "msk_layer_step_tree")
        return st

    def decode_step_tree(self, hidden, kv_cache, cache_len, parents, prev_routing=None, routing_out=None,
                         stream=None, check=True):
        st = msk_decode_step_tree(self.handle, hidden, kv_cache, cache_len, parents, prev_routing, routing_out,
                                  stream)
        if check:
            _check(st, "msk_decode_step_tree")
        return st

    def capture_step(self, hidden, kv_cache, prev_routing=None, routing_out=None):
        """Records one whole step over these buffers as a CUDA graph (see
        msk_step_graph_capture)."""
        _check(msk_step_graph_capture(self.handle, hidden, kv_cache, prev_routing, routing_out),
               "msk_step_graph_capture")

    def replay_step(self, cache_len, parents=None, stream=None, check=True):
        st = msk_step_graph_launch(self.handle, cache_len, parents, stream)
        if check:
            _check(st, "msk_step_graph_launch")
        return st

    def set_timing(self, on):
        _check(load_library().msk_set_timing(self.handle, int(on)), "msk_set_timing")

    def timeline(self):
        """Per-launch, per-block phase timestamps (ns): int64 tensor
        [launches][ctas][TIMELINE_SLOTS] (zeros where a phase was not run)."""
        L = load_library()
        cap = self.n_layers * self.n_ctas * TIMELINE_SLOTS
        buf = (ctypes.c_uint64 * cap)()
        n = ctypes.c_size_t()
        nl = ctypes.c_int32()
        nc = ctypes.c_int32()
        _check(L.msk_get_timeline(self.handle, buf, cap, ctypes.byref(n), ctypes.byref(nl), ctypes.byref(nc)),
               "msk_get_timeline")
        t = torch.tensor(list(buf)[: n.value], dtype=torch.int64)
        return t.reshape(nl.value, nc.value, TIMELINE_SLOTS) if n.value else t

    def set_launch_timing(self, on):
        _check(load_library().msk_set_launch_timing(self.handle, int(on)), "msk_set_launch_timing")

    def launch_ms(self):
        """Durations (ms) of the last call's launches, from CUDA events
        recorded on the call's stream."""
        buf = (ctypes.c_float * self.n_layers)()
        n = ctypes.c_int32()
        _check(load_library().msk_get_launch_ms(self.handle, buf, self.n_layers, ctypes.byref(n)),
               "msk_get_launch_ms")
        return list(buf)[: n.value]

    def set_wait_budget(self, ns):
        _check(load_library().msk_set_wait_budget(self.handle, int(ns)), "msk_set_wait_budget")

    def set_fault_injection(self, barrier, cta):
        _check(load_library().msk_set_fault_injection(self.handle, int(barrier), int(cta)),
               "msk_set_fault_injection")

    def debug_scratch(self, which, out, stream=None):
        """Copies intermediate `which` of the last launch into tensor `out`."""
        n = ctypes.c_size_t()
        _check(load_library().msk_debug_scratch(self.handle, which, _ptr(out), out.numel() * out.element_size(),
                                                ctypes.byref(n), _stream(stream)), "msk_debug_scratch")
        return n.value

    def debug_dequant(self, layer, expert, which, out, stream=None):
        msk_debug_dequant(self.handle, layer, expert, which, out, stream)

    def close(self):
        if getattr(self, "handle", None):
            msk_destroy(self.handle)
            self.handle = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass
