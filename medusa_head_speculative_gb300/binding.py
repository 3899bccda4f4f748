"""ctypes binding of libmedusa.so: the same entry points as include/medusa.h.

Argument marshalling only.  Torch tensors supply device memory and the stream; every step
of the computation runs in the library's CUDA kernels.  There is no fallback: if the
library is missing, loading raises.
"""
from __future__ import annotations

import ctypes as C
import os

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libmedusa.so")

MEDUSA_OK, MEDUSA_ERR_INVALID, MEDUSA_ERR_UNSUPPORTED = 0, -1, -2
MEDUSA_ERR_CUDA, MEDUSA_ERR_DEVICE, MEDUSA_ERR_WORKSPACE = -3, -4, -6
F32, BF16 = 0, 1
GREEDY, TYPICAL, REJECT = 0, 1, 2
MAX_HEADS, MAX_TOPS, MAX_NODES = 8, 16, 256
FLAG_TOKEN_RANGE, FLAG_KV_CAPACITY, FLAG_PAGE_RANGE, FLAG_NONFINITE, FLAG_TIMEOUT = 1, 2, 4, 8, 16
STATUS_NAMES = {0: "OK", -1: "INVALID", -2: "UNSUPPORTED", -3: "CUDA", -4: "DEVICE", -6: "WORKSPACE"}


class MedusaError(RuntimeError):
    def __init__(self, fn, code):
        super().__init__(f"{fn} returned {code} ({STATUS_NAMES.get(code, '?')})")
        self.code = code


class Dims(C.Structure):
    _fields_ = [("B", C.c_int), ("d", C.c_int), ("V", C.c_int), ("K", C.c_int), ("Hq", C.c_int),
                ("Hkv", C.c_int), ("dh", C.c_int), ("dtype", C.c_int), ("rope_base", C.c_float),
                ("capacity", C.c_int), ("page_size", C.c_int), ("num_pages", C.c_int)]


class TreeSpec(C.Structure):
    _fields_ = [("K", C.c_int), ("s", C.c_int * MAX_HEADS), ("N", C.c_int),
                ("parent", C.POINTER(C.c_int32)), ("rank", C.POINTER(C.c_int32))]


class Weights(C.Structure):
    _fields_ = [(n, C.c_void_p) for n in ("w1", "w2", "lm", "emb", "wq", "wk", "wv", "wo")]


class Layer(C.Structure):
    _fields_ = [(n, C.c_void_p) for n in ("wq", "wk", "wv", "wo", "k", "v")]


class KV(C.Structure):
    _fields_ = [("k", C.c_void_p), ("v", C.c_void_p), ("page_table", C.c_void_p),
                ("len", C.c_void_p), ("len_out", C.c_void_p)]


class Accept(C.Structure):
    _fields_ = [("mode", C.c_int), ("temperature", C.c_float), ("eps", C.c_float),
                ("delta", C.c_float), ("uniforms", C.c_void_p)]


class KernelTime(C.Structure):
    _fields_ = [("name", C.c_char * 32), ("launches", C.c_int), ("total_ms", C.c_double)]


class Outputs(C.Structure):
    _fields_ = [("out_tok", C.c_void_p), ("n_acc", C.c_void_p), ("path_nodes", C.c_void_p),
                ("h_next", C.c_void_p), ("root_next", C.c_void_p)]


_lib = None
P = C.c_void_p
SZ = C.c_size_t
I = C.c_int


def lib():
    """Load libmedusa.so (built by medusa_head_speculative_gb300.build)."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(LIB_PATH):
        raise RuntimeError(f"{LIB_PATH} is missing: build it with "
                           "`python -m medusa_head_speculative_gb300.build`")
    L = C.CDLL(LIB_PATH)
    sigs = {
        "medusa_plan_create": (I, [C.POINTER(Dims), C.POINTER(TreeSpec), C.POINTER(P)]),
        "medusa_plan_destroy": (None, [P]),
        "medusa_workspace_size": (SZ, [P]),
        "medusa_get_status": (I, [P, P, C.POINTER(C.c_uint32)]),
        "medusa_step": (I, [P, P, P, C.POINTER(Weights), C.POINTER(KV), Accept,
                            C.POINTER(Outputs), P, SZ, P]),
        "medusa_workspace_size_layers": (SZ, [P, I]),
        "medusa_step_layers": (I, [P, P, P, C.POINTER(Weights), C.POINTER(Layer), I, C.POINTER(KV),
                                   Accept, C.POINTER(Outputs), P, SZ, P]),
        "medusa_heads": (I, [P, P, P, C.POINTER(Weights), P, P, P, P, P, SZ, P]),
        "medusa_heads_noalloc": (I, [P, P, P, C.POINTER(Weights), P, P, P, P]),
        "medusa_tree_build": (I, [P, P, P, P, P, P, P, P, P]),
        "medusa_layer_qkv": (I, [P, C.POINTER(Weights), P, P, P, P, P, P, SZ, P]),
        "medusa_tree_attention": (I, [P, P, C.POINTER(KV), P, P, P, P, P, SZ, P]),
        "medusa_layer_out": (I, [P, C.POINTER(Weights), P, P, P, P, SZ, P]),
        "medusa_verify_logits": (I, [P, C.POINTER(Weights), P, P, Accept, P, P, P, P, SZ, P]),
        "medusa_verify": (I, [P, P, P, P, P, P, P, Accept, C.POINTER(Outputs), P]),
        "medusa_kv_compact": (I, [P, C.POINTER(KV), P, P, P, P, P]),
        "medusa_profile_start": (I, [P, I]),
        "medusa_profile_stop": (I, [P, P, C.POINTER(KernelTime), I, C.POINTER(I), C.POINTER(I)]),
        "medusa_tree_cartesian": (I, [I, C.POINTER(C.c_int), I, C.POINTER(C.c_int32),
                                      C.POINTER(C.c_int32)]),
        "medusa_tree_greedy": (I, [I, C.POINTER(C.c_int), I, C.POINTER(C.c_double), I,
                                   C.POINTER(C.c_int32), C.POINTER(C.c_int32)]),
        "medusa_tree_greedy_device": (I, [I, C.POINTER(C.c_int), I, P, I, P, P, P, P]),
        "medusa_tree_size_choose": (I, [C.POINTER(C.c_double), I, C.POINTER(C.c_int),
                                        C.POINTER(C.c_double), I]),
        "medusa_loop_create": (I, [P, C.POINTER(Weights), C.POINTER(KV), Accept, P, P, P, P, I, P,
                                   SZ, C.POINTER(P)]),
        "medusa_loop_run": (I, [P, I, P]),
        "medusa_loop_steps": (I, [P, P, C.POINTER(C.c_longlong)]),
        "medusa_loop_destroy": (None, [P]),
        "medusa_plan_expire_wait_once": (I, [P, C.c_ulonglong]),
    }
    for name, (res, args) in sigs.items():
        f = getattr(L, name)
        f.restype = res
        f.argtypes = args
    _lib = L
    return L


def _check(fn, code):
    if code != MEDUSA_OK:
        raise MedusaError(fn, code)


def ptr(t):
    """Device (or host) address of a tensor, or None."""
    return None if t is None else t.data_ptr()


def _stream(stream):
    import torch
    s = stream if stream is not None else torch.cuda.current_stream()
    return s.cuda_stream


# ------------------------------------------------------------------ host tree builders
def tree_cartesian(s):
    K = len(s)
    sa = (C.c_int * K)(*s)
    cap = MAX_NODES
    parent = (C.c_int32 * cap)()
    rank = (C.c_int32 * cap)()
    n1 = lib().medusa_tree_cartesian(K, sa, cap, parent, rank)
    if n1 < 0:
        raise MedusaError("medusa_tree_cartesian", n1)
    return np.array(parent[:n1], dtype=np.int32), np.array(rank[:n1], dtype=np.int32)


def tree_greedy(s, a, N):
    a = np.ascontiguousarray(a, dtype=np.float64)
    K, smax = a.shape
    sa = (C.c_int * K)(*s)
    parent = (C.c_int32 * (N + 1))()
    rank = (C.c_int32 * (N + 1))()
    n1 = lib().medusa_tree_greedy(K, sa, smax, a.ctypes.data_as(C.POINTER(C.c_double)), N,
                                  parent, rank)
    if n1 < 0:
        raise MedusaError("medusa_tree_greedy", n1)
    return np.array(parent[:n1], dtype=np.int32), np.array(rank[:n1], dtype=np.int32)


def tree_greedy_device(s, a_dev, N, parent, rank, expected=None, stream=None):
    """medusa_tree_greedy_device: a_dev a [K][smax] float64 CUDA tensor; parent, rank int32
    CUDA tensors of N+1 entries, expected float64 (N+1) or None."""
    K, smax = a_dev.shape
    sa = (C.c_int * K)(*s)
    _check("medusa_tree_greedy_device",
           lib().medusa_tree_greedy_device(K, sa, smax, ptr(a_dev), N, ptr(parent), ptr(rank),
                                           ptr(expected), _stream(stream)))


def tree_size_choose(expected, sizes, step_ms):
    """medusa_tree_size_choose: index into sizes of the best expected tokens per time."""
    e = np.ascontiguousarray(expected, dtype=np.float64)
    sz = (C.c_int * len(sizes))(*sizes)
    ms = np.ascontiguousarray(step_ms, dtype=np.float64)
    i = lib().medusa_tree_size_choose(e.ctypes.data_as(C.POINTER(C.c_double)), len(e) - 1, sz,
                                      ms.ctypes.data_as(C.POINTER(C.c_double)), len(sizes))
    if i < 0:
        raise MedusaError("medusa_tree_size_choose", i)
    return i


# ------------------------------------------------------------------ plan
class Plan:
    """Owns a medusa_plan: validated sizes and the uploaded tree spec."""

    def __init__(self, B, d, V, K, Hq, Hkv, dh, dtype, capacity, s, parent, rank,
                 rope_base=10000.0, page_size=0, num_pages=0):
        self.dims = Dims(B, d, V, K, Hq, Hkv, dh, dtype, rope_base, capacity, page_size, num_pages)
        parent = np.ascontiguousarray(parent, dtype=np.int32)
        rank = np.ascontiguousarray(rank, dtype=np.int32)
        self.spec = TreeSpec()
        self.spec.K = K
        for k in range(MAX_HEADS):
            self.spec.s[k] = int(s[k]) if k < len(s) else 0
        self.spec.N = len(parent) - 1
        self._keep = (parent, rank)
        self.spec.parent = parent.ctypes.data_as(C.POINTER(C.c_int32))
        self.spec.rank = rank.ctypes.data_as(C.POINTER(C.c_int32))
        h = P()
        _check("medusa_plan_create", lib().medusa_plan_create(C.byref(self.dims), C.byref(self.spec),
                                                              C.byref(h)))
        self.handle = h
        self.B, self.d, self.V, self.K, self.N = B, d, V, K, len(parent) - 1
        self.Hq, self.Hkv, self.dh, self.dtype = Hq, Hkv, dh, dtype
        self.n1 = self.N + 1
        self.parent, self.rank = parent, rank

    @property
    def workspace_size(self):
        return lib().medusa_workspace_size(self.handle)

    def workspace_size_layers(self, n_layers):
        return lib().medusa_workspace_size_layers(self.handle, n_layers)

    def status(self, stream=None):
        flags = C.c_uint32(0)
        code = lib().medusa_get_status(self.handle, _stream(stream), C.byref(flags))
        if code not in (MEDUSA_OK, MEDUSA_ERR_DEVICE):
            raise MedusaError("medusa_get_status", code)
        return flags.value

    def expire_wait_once(self, ns):
        """Failure-path testing: the next verification-logit GEMM's wait runs out after ns."""
        _check("medusa_plan_expire_wait_once", lib().medusa_plan_expire_wait_once(self.handle, int(ns)))

    def profile_start(self, max_launches):
        _check("medusa_profile_start", lib().medusa_profile_start(self.handle, max_launches))

    def profile_stop(self, stream=None):
        """Per-kernel {name: (launches, total_ms)} in first-launch order, and the launch count."""
        out = (KernelTime * 64)()
        n, launches = C.c_int(0), C.c_int(0)
        _check("medusa_profile_stop", lib().medusa_profile_stop(self.handle, _stream(stream), out, 64,
                                                                C.byref(n), C.byref(launches)))
        return {out[i].name.decode(): (out[i].launches, out[i].total_ms) for i in range(n.value)}, \
            launches.value

    def close(self):
        if getattr(self, "handle", None):
            lib().medusa_plan_destroy(self.handle)
            self.handle = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass


def weights_struct(w):
    return Weights(*(ptr(w.get(n)) for n in ("w1", "w2", "lm", "emb", "wq", "wk", "wv", "wo")))


def layers_array(layers):
    """ctypes array of Layer from dicts with wq, wk, wv, wo, k, v (device tensors)."""
    arr = (Layer * len(layers))()
    for i, L in enumerate(layers):
        arr[i] = Layer(*(ptr(L[n]) for n in ("wq", "wk", "wv", "wo", "k", "v")))
    return arr


def kv_struct(k, v, length, len_out=None, page_table=None):
    return KV(ptr(k), ptr(v), ptr(page_table), ptr(length), ptr(len_out))


def accept_struct(mode="greedy", temperature=0.0, eps=0.09, delta=0.3, uniforms=None):
    code = {"typical": TYPICAL, "reject": REJECT}.get(mode, GREEDY)
    return Accept(code, temperature, eps, delta, ptr(uniforms))


def outputs_struct(out_tok, n_acc, path_nodes, h_next, root_next):
    return Outputs(ptr(out_tok), ptr(n_acc), ptr(path_nodes), ptr(h_next), ptr(root_next))


# ------------------------------------------------------------------ entry points
def step(plan, h, root_in, wts, kv, accept, outs, ws, stream=None):
    _check("medusa_step", lib().medusa_step(plan.handle, ptr(h), ptr(root_in), C.byref(wts),
                                            C.byref(kv), accept, C.byref(outs), ptr(ws),
                                            ws.numel() * ws.element_size(), _stream(stream)))


def step_layers(plan, h, root_in, wts, layers, kv, accept, outs, ws, stream=None):
    """medusa_step_layers; `layers` from layers_array."""
    _check("medusa_step_layers",
           lib().medusa_step_layers(plan.handle, ptr(h), ptr(root_in), C.byref(wts), layers,
                                    len(layers), C.byref(kv), accept, C.byref(outs), ptr(ws),
                                    ws.numel() * ws.element_size(), _stream(stream)))


def heads(plan, h, root_in, wts, logits, topk_tok, topk_val, root, ws, stream=None):
    _check("medusa_heads", lib().medusa_heads(plan.handle, ptr(h), ptr(root_in), C.byref(wts),
                                              ptr(logits), ptr(topk_tok), ptr(topk_val), ptr(root),
                                              ptr(ws), ws.numel() * ws.element_size(),
                                              _stream(stream)))


def heads_noalloc(plan, h, root_in, wts, topk_tok, topk_val, root, stream=None):
    """Heads stage with no workspace: scratch in the library's fixed device array."""
    _check("medusa_heads_noalloc", lib().medusa_heads_noalloc(plan.handle, ptr(h), ptr(root_in),
                                                              C.byref(wts), ptr(topk_tok),
                                                              ptr(topk_val), ptr(root),
                                                              _stream(stream)))


def tree_build(plan, topk_tok, root, length, tok, pos, mask, retrieve, stream=None):
    _check("medusa_tree_build", lib().medusa_tree_build(plan.handle, ptr(topk_tok), ptr(root),
                                                        ptr(length), ptr(tok), ptr(pos), ptr(mask),
                                                        ptr(retrieve), _stream(stream)))


def layer_qkv(plan, wts, tok, pos, q, tk, tv, ws, stream=None):
    _check("medusa_layer_qkv", lib().medusa_layer_qkv(plan.handle, C.byref(wts), ptr(tok), ptr(pos),
                                                      ptr(q), ptr(tk), ptr(tv), ptr(ws),
                                                      ws.numel() * ws.element_size(),
                                                      _stream(stream)))


def tree_attention(plan, q, kv, tk, tv, mask, o, ws, stream=None):
    _check("medusa_tree_attention",
           lib().medusa_tree_attention(plan.handle, ptr(q), C.byref(kv), ptr(tk), ptr(tv), ptr(mask),
                                       ptr(o), ptr(ws), ws.numel() * ws.element_size(),
                                       _stream(stream)))


def layer_out(plan, wts, tok, o, hprime, ws, stream=None):
    _check("medusa_layer_out", lib().medusa_layer_out(plan.handle, C.byref(wts), ptr(tok), ptr(o),
                                                      ptr(hprime), ptr(ws),
                                                      ws.numel() * ws.element_size(),
                                                      _stream(stream)))


def verify_logits(plan, wts, hprime, tok, accept, logits, am, stats, ws, stream=None):
    _check("medusa_verify_logits",
           lib().medusa_verify_logits(plan.handle, C.byref(wts), ptr(hprime), ptr(tok), accept,
                                      ptr(logits), ptr(am), ptr(stats), ptr(ws),
                                      ws.numel() * ws.element_size(), _stream(stream)))


def verify(plan, tok, am, stats, retrieve, hprime, accept, outs, stream=None, logits=None):
    _check("medusa_verify", lib().medusa_verify(plan.handle, ptr(tok), ptr(am), ptr(stats),
                                                ptr(logits), ptr(retrieve), ptr(hprime), accept,
                                                C.byref(outs), _stream(stream)))


def kv_compact(plan, kv, tk, tv, path_nodes, n_acc, stream=None):
    _check("medusa_kv_compact", lib().medusa_kv_compact(plan.handle, C.byref(kv), ptr(tk), ptr(tv),
                                                        ptr(path_nodes), ptr(n_acc),
                                                        _stream(stream)))


class Loop:
    """Owns a medusa_loop: one medusa_step with its state carried in place (h, root, cache
    lengths) plus the append to the token rings, captured once as a CUDA graph.  The
    tensors passed here must outlive the loop (its replays use their addresses)."""

    def __init__(self, plan, wts, kv, accept, h, root, tokens, n_acc, ws):
        self._keep = (plan, wts, kv, h, root, tokens, n_acc, ws)
        self.max_steps = tokens.shape[0]
        out = P()
        _check("medusa_loop_create",
               lib().medusa_loop_create(plan.handle, C.byref(wts), C.byref(kv), accept, ptr(h),
                                        ptr(root), ptr(tokens), ptr(n_acc), self.max_steps,
                                        ptr(ws), ws.numel() * ws.element_size(), C.byref(out)))
        self.handle = out

    def run(self, n_steps, stream=None):
        _check("medusa_loop_run", lib().medusa_loop_run(self.handle, int(n_steps), _stream(stream)))

    def steps(self, stream=None):
        n = C.c_longlong(0)
        _check("medusa_loop_steps", lib().medusa_loop_steps(self.handle, _stream(stream), C.byref(n)))
        return n.value

    def close(self):
        if getattr(self, "handle", None):
            lib().medusa_loop_destroy(self.handle)
            self.handle = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass

