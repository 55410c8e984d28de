"""Thin ctypes binding of libmk.so (include/mk.h).

The functions below carry the C ABI's names and only marshal arguments: torch
tensors become device pointers, dicts become the config/weights structs.  Every
step of the decode path runs in the library's CUDA kernels; if the library is
missing this module raises instead of falling back to anything else.
"""
from __future__ import annotations

import ctypes
import os

import numpy as np

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "libmk.so")

MK_OK, MK_ERR_INVALID, MK_ERR_UNSUPPORTED, MK_ERR_CUDA, MK_ERR_OOM = 0, 1, 2, 3, 4
MK_ERR_TIMEOUT, MK_ERR_BAD_PAGE, MK_ERR_BAD_TOKEN, MK_ERR_STATE, MK_ERR_NAN = 5, 6, 7, 8, 9
STATUS_NAMES = {0: "MK_OK", 1: "MK_ERR_INVALID", 2: "MK_ERR_UNSUPPORTED", 3: "MK_ERR_CUDA",
                4: "MK_ERR_OOM", 5: "MK_ERR_TIMEOUT", 6: "MK_ERR_BAD_PAGE",
                7: "MK_ERR_BAD_TOKEN", 8: "MK_ERR_STATE", 9: "MK_ERR_NAN"}

MK_READ_HIDDEN, MK_READ_ROUTES, MK_READ_ROUTE_W, MK_READ_ACTIVE = 1, 2, 3, 4
MK_READ_SEQ_LENS, MK_READ_COUNTERS, MK_READ_ROUTER_LOGITS, MK_READ_TRACE_COUNT = 5, 6, 7, 8
MK_READ_FINAL_COUNTERS, MK_READ_FINAL_QUEUES, MK_READ_TASKS = 9, 10, 11
MK_EXPERT_BF16, MK_EXPERT_FP8, MK_WEIGHTS_FP8 = 0, 1, 2
(MK_Q_NUM_SMS, MK_Q_NUM_TASKS, MK_Q_NUM_COUNTERS, MK_Q_PACKED_BYTES, MK_Q_MAX_ACTIVE,
 MK_Q_SPLIT_PAGES, MK_Q_SMEM_BYTES, MK_Q_PEROP_LAUNCHES, MK_Q_THREADS, MK_Q_STAGE_BYTES,
 MK_Q_NUM_STAGES, MK_Q_TENSOR_CORES) = range(1, 13)

# exported symbols (kept equal to the declarations of include/mk.h)
EXPORTS = ["mk_create", "mk_plan", "mk_decode_step", "mk_decode_steps", "mk_decode_step_host", "mk_decode_step_noalloc",
           "mk_decode_step_perop", "mk_get_status", "mk_set_fixed", "mk_set_deterministic", "mk_set_inspect", "mk_set_trace",
           "mk_plan_drop_signal", "mk_read", "mk_read_expert_fp8", "mk_read_weight_fp8", "mk_query",
           "mk_plan_dry", "mk_last_error", "mk_destroy", "mk_version"]


class MkError(RuntimeError):
    def __init__(self, code, msg):
        super().__init__(f"{STATUS_NAMES.get(code, code)}: {msg}")
        self.code = code


class mk_config(ctypes.Structure):
    _fields_ = [("n_layers", ctypes.c_int32), ("d_model", ctypes.c_int32),
                ("n_q_heads", ctypes.c_int32), ("n_kv_heads", ctypes.c_int32),
                ("head_dim", ctypes.c_int32), ("n_experts", ctypes.c_int32),
                ("top_k", ctypes.c_int32), ("d_ff", ctypes.c_int32), ("vocab", ctypes.c_int32),
                ("page_size", ctypes.c_int32), ("max_batch", ctypes.c_int32),
                ("sliding_window", ctypes.c_int32), ("swa_layer_mask", ctypes.c_uint64),
                ("rope_theta", ctypes.c_float), ("rms_eps", ctypes.c_float),
                ("timeout_ms", ctypes.c_int32), ("dense_layer_mask", ctypes.c_uint64),
                ("dense_ff", ctypes.c_int32), ("expert_dtype", ctypes.c_int32)]


_PP = ctypes.POINTER(ctypes.c_void_p)


class mk_weights(ctypes.Structure):
    _fields_ = [("embed", ctypes.c_void_p), ("lm_head", ctypes.c_void_p),
                ("final_norm", ctypes.c_void_p), ("attn_norm", _PP), ("wq", _PP), ("wk", _PP),
                ("wv", _PP), ("wo", _PP), ("router", _PP), ("w_gate", _PP), ("w_up", _PP),
                ("w_down", _PP), ("ffn_gate", _PP), ("ffn_up", _PP), ("ffn_down", _PP)]


class mk_error_info(ctypes.Structure):
    _fields_ = [("code", ctypes.c_int32), ("task", ctypes.c_int32), ("counter", ctypes.c_int32),
                ("observed", ctypes.c_int32), ("target", ctypes.c_int32), ("sm", ctypes.c_int32)]


_lib = None


def load_library(path: str = LIB_PATH) -> ctypes.CDLL:
    """Load libmk.so; raises if it has not been built (no fallback path exists)."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(path):
        raise ImportError(f"{path} is missing: build it with "
                          "`python -m persistent_moe_decode_cta_gb300.build`")
    lib = ctypes.CDLL(path)
    vp, i32, sz = ctypes.c_void_p, ctypes.c_int, ctypes.c_size_t
    H = ctypes.c_void_p
    lib.mk_create.argtypes = [ctypes.POINTER(mk_config), ctypes.POINTER(mk_weights), vp,
                              ctypes.POINTER(H)]
    lib.mk_plan.argtypes = [H, i32, ctypes.POINTER(ctypes.c_int32), vp, i32, i32]
    lib.mk_decode_step.argtypes = [H, vp, vp, vp, vp, vp]
    lib.mk_decode_steps.argtypes = [H, vp, i32, vp, vp, vp, vp, vp]
    lib.mk_decode_step_host.argtypes = [H, vp, vp, vp, vp, vp]
    lib.mk_decode_step_noalloc.argtypes = [H, vp, vp, vp, vp, vp]
    lib.mk_decode_step_perop.argtypes = [H, vp, vp, vp, vp, vp, i32]
    lib.mk_get_status.argtypes = [H, ctypes.POINTER(mk_error_info)]
    lib.mk_set_fixed.argtypes = [H, i32]
    lib.mk_set_deterministic.argtypes = [H, i32]
    lib.mk_set_inspect.argtypes = [H, i32]
    lib.mk_set_trace.argtypes = [H, vp, i32]
    lib.mk_plan_drop_signal.argtypes = [H, i32]
    lib.mk_read.argtypes = [H, i32, vp, sz]
    lib.mk_read_expert_fp8.argtypes = [H, i32, i32, vp, sz]
    lib.mk_read_weight_fp8.argtypes = [H, i32, i32, vp, sz]
    lib.mk_query.argtypes = [H, i32, ctypes.POINTER(ctypes.c_int64)]
    lib.mk_plan_dry.argtypes = [ctypes.POINTER(mk_config), i32, i32, vp, i32, vp, vp, i32, vp]
    lib.mk_last_error.argtypes = [H]
    lib.mk_last_error.restype = ctypes.c_char_p
    lib.mk_destroy.argtypes = [H]
    lib.mk_destroy.restype = None
    lib.mk_version.argtypes = []
    for name in EXPORTS:
        if name not in ("mk_last_error", "mk_destroy"):
            getattr(lib, name).restype = ctypes.c_int
    _lib = lib
    return lib


def _check(rc, handle=None):
    if rc != MK_OK:
        msg = load_library().mk_last_error(handle)
        raise MkError(rc, msg.decode() if msg else "")
    return rc


def make_config(cfg: dict, max_batch: int = 8, timeout_ms: int = 2000) -> mk_config:
    mask = 0
    for l in cfg.get("swa_layers", ()):
        mask |= 1 << int(l)
    dense = 0
    for l in cfg.get("dense_layers", ()):
        dense |= 1 << int(l)
    return mk_config(cfg["n_layers"], cfg["d_model"], cfg["n_q_heads"], cfg["n_kv_heads"],
                     cfg["head_dim"], cfg["n_experts"], cfg["top_k"], cfg["d_ff"], cfg["vocab"],
                     cfg.get("page_size", 16), max_batch, cfg.get("sliding_window", 0), mask,
                     cfg["rope_theta"], cfg["rms_eps"], timeout_ms, dense,
                     cfg.get("dense_ff", 0) if dense else 0,
                     MK_WEIGHTS_FP8 if cfg.get("dense_dtype", "bf16") == "fp8"
                     else MK_EXPERT_FP8 if cfg.get("expert_dtype", "bf16") == "fp8" else MK_EXPERT_BF16)


def _ptrs(t, n):
    """Device pointers of the n leading slices of a stacked tensor."""
    base, stride = t.data_ptr(), t.stride(0) * t.element_size()
    return (ctypes.c_void_p * n)(*[base + i * stride for i in range(n)])


def make_weights(W: dict, cfg: dict):
    """mk_weights from the stacked bf16 tensors of synth.make_weights (device tensors).
    Returns (struct, keepalive)."""
    L, E = cfg["n_layers"], cfg["n_experts"]
    for k, t in W.items():
        if not t.is_cuda or not t.is_contiguous():
            raise ValueError(f"weight {k} must be a contiguous CUDA tensor")
    arrs = dict(attn_norm=_ptrs(W["attn_norm"], L), wq=_ptrs(W["wq"], L), wk=_ptrs(W["wk"], L),
                wv=_ptrs(W["wv"], L), wo=_ptrs(W["wo"], L), router=_ptrs(W["router"], L),
                w_gate=_ptrs(W["w_gate"].view(L * E, *W["w_gate"].shape[2:]), L * E),
                w_up=_ptrs(W["w_up"].view(L * E, *W["w_up"].shape[2:]), L * E),
                w_down=_ptrs(W["w_down"].view(L * E, *W["w_down"].shape[2:]), L * E))
    names = ["attn_norm", "wq", "wk", "wv", "wo", "router", "w_gate", "w_up", "w_down"]
    if "ffn_gate" in W:  # the dense FFNs of a mixed stack
        for k in ("ffn_gate", "ffn_up", "ffn_down"):
            arrs[k] = _ptrs(W[k], L)
        names += ["ffn_gate", "ffn_up", "ffn_down"]
    s = mk_weights(W["embed"].data_ptr(), W["lm_head"].data_ptr(), W["final_norm"].data_ptr(),
                   *[ctypes.cast(arrs[k], _PP) for k in names])
    return s, arrs


def _stream_ptr(stream):
    if stream is None:
        import torch
        return torch.cuda.current_stream().cuda_stream
    return getattr(stream, "cuda_stream", stream)


# ---------------------------------------------------------------- C ABI wrappers

def mk_create(cfg: dict, W: dict, max_batch: int = 8, timeout_ms: int = 2000, stream=None):
    lib = load_library()
    c = make_config(cfg, max_batch, timeout_ms)
    w, keep = make_weights(W, cfg)
    h = ctypes.c_void_p()
    _check(lib.mk_create(ctypes.byref(c), ctypes.byref(w), _stream_ptr(stream), ctypes.byref(h)))
    del keep
    return h


def mk_plan(h, seq_lens, page_table, n_pages: int):
    """page_table: int32 CUDA tensor [B, max_pages]."""
    sl = (ctypes.c_int32 * len(seq_lens))(*[int(x) for x in seq_lens])
    if page_table.dtype.itemsize != 4 or not page_table.is_cuda or not page_table.is_contiguous():
        raise ValueError("page_table must be a contiguous int32 CUDA tensor")
    _check(load_library().mk_plan(h, len(seq_lens), sl, page_table.data_ptr(),
                                  page_table.shape[1], int(n_pages)), h)


def mk_decode_step(h, tokens, k_cache, v_cache, logits, stream=None):
    _check(load_library().mk_decode_step(h, tokens.data_ptr(), k_cache.data_ptr(),
                                         v_cache.data_ptr(), logits.data_ptr(),
                                         _stream_ptr(stream)), h)


def mk_decode_steps(h, tokens, n_steps, k_cache, v_cache, logits, tokens_out, stream=None):
    """n_steps greedy steps in one launch; tokens_out: device int32 [n_steps, batch]."""
    _check(load_library().mk_decode_steps(h, tokens.data_ptr(), int(n_steps), k_cache.data_ptr(),
                                          v_cache.data_ptr(), logits.data_ptr(), tokens_out.data_ptr(),
                                          _stream_ptr(stream)), h)


def mk_decode_step_noalloc(h, tokens, k_cache, v_cache, logits, stream=None):
    """mk_decode_step with the step scratch in the library's static device buffer."""
    _check(load_library().mk_decode_step_noalloc(h, tokens.data_ptr(), k_cache.data_ptr(),
                                                 v_cache.data_ptr(), logits.data_ptr(),
                                                 _stream_ptr(stream)), h)


def mk_decode_step_host(h, tokens_host, k_cache, v_cache, logits_host, stream=None):
    """tokens_host / logits_host: CPU tensors (pinned for asynchronous copies)."""
    _check(load_library().mk_decode_step_host(h, tokens_host.data_ptr(), k_cache.data_ptr(),
                                              v_cache.data_ptr(), logits_host.data_ptr(),
                                              _stream_ptr(stream)), h)


def mk_decode_step_perop(h, tokens, k_cache, v_cache, logits, use_graph=False, stream=None):
    _check(load_library().mk_decode_step_perop(h, tokens.data_ptr(), k_cache.data_ptr(),
                                               v_cache.data_ptr(), logits.data_ptr(),
                                               _stream_ptr(stream), int(bool(use_graph))), h)


def mk_get_status(h) -> dict:
    info = mk_error_info()
    load_library().mk_get_status(h, ctypes.byref(info))
    return {k: getattr(info, k) for k, _ in mk_error_info._fields_}


def mk_set_fixed(h, fixed: bool):
    _check(load_library().mk_set_fixed(h, int(bool(fixed))), h)


def mk_set_deterministic(h, on: bool):
    _check(load_library().mk_set_deterministic(h, int(bool(on))), h)


def mk_set_inspect(h, on: bool):
    _check(load_library().mk_set_inspect(h, int(bool(on))), h)


def mk_plan_drop_signal(h, task: int):
    _check(load_library().mk_plan_drop_signal(h, int(task)), h)


def mk_set_trace(h, records, capacity: int):
    """records: uint64/int64 CUDA tensor [capacity, 16] (or None with capacity 0)."""
    _check(load_library().mk_set_trace(h, records.data_ptr() if records is not None else None,
                                       int(capacity)), h)


def mk_read(h, what: int, shape, dtype) -> np.ndarray:
    out = np.empty(shape, dtype=dtype)
    _check(load_library().mk_read(h, what, out.ctypes.data, out.nbytes), h)
    return out


def mk_read_expert_fp8(h, layer: int, expert: int, d_model: int, d_ff: int) -> dict:
    """The stored FP8 form of one routed expert, row-major: codes (uint8) and scales
    (float32, one per row) of gate [d_ff, d_model], up [d_ff, d_model] and down
    [d_model, d_ff]."""
    d, f = int(d_model), int(d_ff)
    n = 3 * f * d + 4 * (2 * f + d)
    buf = np.empty(n, dtype=np.uint8)
    _check(load_library().mk_read_expert_fp8(h, int(layer), int(expert), buf.ctypes.data, n), h)
    o = 0
    out = {}
    for name, shape in (("gate", (f, d)), ("up", (f, d)), ("down", (d, f))):
        out[name + "_codes"] = buf[o:o + f * d].reshape(shape)
        o += f * d
    for name, shape in (("gate", (f,)), ("up", (f,)), ("down", (d,))):
        k = int(np.prod(shape))
        out[name + "_scales"] = buf[o:o + 4 * k].view(np.float32).reshape(shape)
        o += 4 * k
    return out


MK_W_Q, MK_W_K, MK_W_V, MK_W_O, MK_W_LM = 0, 1, 2, 3, 4


def mk_read_weight_fp8(h, matrix: int, layer: int, rows: int, cols: int):
    """The stored FP8 form of a projection: (codes uint8 [rows, cols], scales float32 [rows])."""
    n = rows * cols + 4 * rows
    buf = np.empty(n, dtype=np.uint8)
    _check(load_library().mk_read_weight_fp8(h, int(matrix), int(layer), buf.ctypes.data, n), h)
    return buf[:rows * cols].reshape(rows, cols), buf[rows * cols:].view(np.float32)


def mk_query(h, what: int) -> int:
    v = ctypes.c_int64()
    _check(load_library().mk_query(h, what, ctypes.byref(v)), h)
    return v.value


def mk_plan_dry(cfg: dict, batch: int, n_sms: int, max_batch: int = 8):
    """Host-only plan: (tasks [n,32], sm_off [n_sms+1], sm_list, info[32])."""
    lib = load_library()
    c = make_config(cfg, max_batch)
    info = np.zeros(32, dtype=np.int32)
    rc = lib.mk_plan_dry(ctypes.byref(c), batch, n_sms, None, 0, None, None, 0,
                         info.ctypes.data)
    n_tasks, n_list = int(info[0]), int(info[1])
    if n_tasks <= 0:
        _check(rc if rc != MK_OK else MK_ERR_INVALID)
    tasks = np.zeros((n_tasks, 32), dtype=np.int32)
    sm_off = np.zeros(n_sms + 1, dtype=np.int32)
    sm_list = np.zeros(max(n_list, 1), dtype=np.int32)
    _check(lib.mk_plan_dry(ctypes.byref(c), batch, n_sms, tasks.ctypes.data, n_tasks,
                           sm_off.ctypes.data, sm_list.ctypes.data, len(sm_list),
                           info.ctypes.data))
    return tasks, sm_off, sm_list[:n_list], info


def mk_destroy(h):
    if h:
        load_library().mk_destroy(h)


# ---------------------------------------------------------------- convenience object

class Megakernel:
    """Owns an mk handle: create (pack weights) -> plan(batch) -> step()..."""

    def __init__(self, cfg: dict, W: dict, max_batch: int = 8, timeout_ms: int = 2000):
        self.cfg = dict(cfg)
        self.max_batch = max_batch
        self.h = mk_create(cfg, W, max_batch, timeout_ms)
        self.B = 0

    def plan(self, seq_lens, page_table, n_pages):
        mk_plan(self.h, seq_lens, page_table, n_pages)
        self.B = len(seq_lens)
        # every step reads the page table through the pointer given here: hold the
        # tensor so that its memory is not recycled while the plan is in use
        self._page_table = page_table

    def step(self, tokens, k_cache, v_cache, logits, stream=None):
        mk_decode_step(self.h, tokens, k_cache, v_cache, logits, stream)

    def steps(self, tokens, n_steps, k_cache, v_cache, logits, tokens_out=None, stream=None):
        """n_steps greedy decode steps in one launch (device-side token feedback).
        Returns the int32 [n_steps, batch] tensor of each step's greedy token."""
        import torch
        if tokens_out is None:
            tokens_out = torch.empty(n_steps, tokens.shape[0], dtype=torch.int32, device=tokens.device)
        mk_decode_steps(self.h, tokens, n_steps, k_cache, v_cache, logits, tokens_out, stream)
        return tokens_out

    def step_host(self, tokens_host, k_cache, v_cache, logits_host, stream=None):
        mk_decode_step_host(self.h, tokens_host, k_cache, v_cache, logits_host, stream)

    def step_perop(self, tokens, k_cache, v_cache, logits, use_graph=False, stream=None):
        mk_decode_step_perop(self.h, tokens, k_cache, v_cache, logits, use_graph, stream)

    def status(self):
        return mk_get_status(self.h)

    def set_fixed(self, fixed=True):
        mk_set_fixed(self.h, fixed)

    def set_deterministic(self, on=True):
        """Deterministic steps from the next plan() on (fixed-point layer accumulators)."""
        mk_set_deterministic(self.h, on)

    def trace_on(self, capacity=1 << 20):
        import torch
        self._trace = torch.zeros((capacity, 16), dtype=torch.int64, device="cuda")
        mk_set_trace(self.h, self._trace, capacity)

    def trace_off(self):
        mk_set_trace(self.h, None, 0)
        self._trace = None

    def trace_records(self):
        """int64 array [n, 16] of the records appended since trace_on()."""
        n = int(mk_read(self.h, MK_READ_TRACE_COUNT, (1,), np.uint32)[0])
        n = min(n, self._trace.shape[0])
        return self._trace[:n].cpu().numpy()

    def query(self, what):
        return mk_query(self.h, what)

    def hidden(self):
        c = self.cfg
        return mk_read(self.h, MK_READ_HIDDEN, (c["n_layers"] + 1, self.B, c["d_model"]), np.float32)

    def expert_fp8(self, layer: int, expert: int) -> dict:
        c = self.cfg
        return mk_read_expert_fp8(self.h, layer, expert, c["d_model"], c["d_ff"])

    def weight_fp8(self, matrix: int, layer: int = 0):
        c = self.cfg
        d, hq, hkv, hd = c["d_model"], c["n_q_heads"], c["n_kv_heads"], c["head_dim"]
        rows, cols = {MK_W_Q: (hq * hd, d), MK_W_K: (hkv * hd, d), MK_W_V: (hkv * hd, d),
                      MK_W_O: (d, hq * hd), MK_W_LM: (c["vocab"], d)}[matrix]
        return mk_read_weight_fp8(self.h, matrix, layer, rows, cols)

    def routes(self):
        c = self.cfg
        idx = mk_read(self.h, MK_READ_ROUTES, (c["n_layers"], self.B, c["top_k"]), np.int32)
        w = mk_read(self.h, MK_READ_ROUTE_W, (c["n_layers"], self.B, c["top_k"]), np.float32)
        return idx, w

    def router_logits(self):
        c = self.cfg
        return mk_read(self.h, MK_READ_ROUTER_LOGITS, (c["n_layers"], self.B, c["n_experts"]),
                       np.float32)

    def active(self):
        """Per layer: list of (expert, [(b, j), ...]) in slot order."""
        c = self.cfg
        maxa = self.query(MK_Q_MAX_ACTIVE)
        per = 1 + maxa * (2 + self.B)
        raw = mk_read(self.h, MK_READ_ACTIVE, (c["n_layers"], per), np.int32)
        out = []
        for l in range(c["n_layers"]):
            r = raw[l]
            lst = []
            for a in range(int(r[0])):
                q = r[1 + a * (2 + self.B):]
                lst.append((int(q[0]), [(int(v) >> 4, int(v) & 15) for v in q[2:2 + int(q[1])]]))
            out.append(lst)
        return out

    def seq_lens(self):
        return mk_read(self.h, MK_READ_SEQ_LENS, (self.B,), np.int32)

    def counters(self):
        return mk_read(self.h, MK_READ_COUNTERS, (self.query(MK_Q_NUM_COUNTERS),), np.uint32)

    def inspect(self, on=True):
        mk_set_inspect(self.h, on)

    def final_counters(self):
        """Every counter's value at the end of the last inspected step (before reset)."""
        return mk_read(self.h, MK_READ_FINAL_COUNTERS, (self.query(MK_Q_NUM_COUNTERS),), np.uint32)

    def final_queues(self):
        """(heads, counts), each int32 [3 * n_layers], at the end of the last inspected step."""
        q = mk_read(self.h, MK_READ_FINAL_QUEUES, (2, 3 * self.cfg["n_layers"]), np.int32)
        return q[0], q[1]

    def tasks(self):
        """The plan's descriptor table, int32 [n_tasks, 32]."""
        return mk_read(self.h, MK_READ_TASKS, (self.query(MK_Q_NUM_TASKS), 32), np.int32)

    def close(self):
        if self.h:
            mk_destroy(self.h)
            self.h = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass
