"""ctypes binding of libspecng (the C ABI declared in include/specng.h).

Argument marshalling only: every step of the path runs in the library's
CUDA kernels.  Tensors must be contiguous CUDA tensors of the stated dtype;
calls are enqueued on the current torch stream of the tensors' device.
There is no CPU fallback: if the library is missing, loading fails loudly.
"""
from __future__ import annotations

import ctypes
import os
from dataclasses import dataclass
from typing import Optional

import torch

# The library to load: libspecng.so next to this file, or the build named by
# SPECNG_LIBRARY (e.g. libspecng_checked.so, the index-checked build).
_LIB_PATH = os.environ.get("SPECNG_LIBRARY") or os.path.join(os.path.dirname(os.path.abspath(__file__)),
                                                              "libspecng.so")

SPECNG_OK = 0
SPECNG_F32 = 0
SPECNG_BF16 = 1

STATUS_BITS = {
    0x01: "TABLE_FULL",
    0x02: "TOKEN_OOR",
    0x04: "NONFINITE",
    0x08: "HIST_OVERFLOW",
    0x10: "BAD_K",
    0x20: "COUNT_SAT",
    0x40: "HIST_SHRANK",
    0x80: "TIMEOUT",
    0x100: "CHECKED_OOB",
    0x200: "KV_SHORT",
}

# Every symbol include/specng.h declares.
EXPORTED = (
    "specng_ngram_create", "specng_ngram_destroy", "specng_ngram_reset", "specng_ngram_capacity",
    "specng_ngram_set_min_count",
    "ngram_update", "ngram_draft", "spec_verify_workspace_bytes", "spec_verify_workspace_init",
    "spec_verify", "spec_verify_noalloc", "spec_verify_lmhead_workspace_bytes", "spec_verify_lmhead", "spec_append", "spec_commit", "specng_get_status", "specng_strerror",
    "specng_last_error", "specng_philox4x32_10", "specng_set_verify_marker", "specng_get_counters",
    "specng_kv_init", "specng_kv_reserve", "specng_kv_trim", "specng_kv_release", "specng_step_advance",
)

# Diagnostic counters (SPECNG_DIAG_*): runs of the exact (fp64) paths.
DIAG = {"accept_f64": 0, "sample_f64": 1, "residual_f64": 2, "greedy_f64": 3, "residual_zero": 4}
DIAG_N = 8


class SpecngError(RuntimeError):
    pass


class VerifyParamsC(ctypes.Structure):
    _fields_ = [
        ("temperature", ctypes.c_float),
        ("softcap", ctypes.c_float),
        ("rep_penalty", ctypes.c_float),
        ("rep_window", ctypes.c_int32),
        ("ema_tau", ctypes.c_float),
        ("ema_thresh", ctypes.c_float),
        ("gate_enabled", ctypes.c_int32),
        ("pad_", ctypes.c_uint32),
        ("seed", ctypes.c_uint64),
        ("step", ctypes.c_uint64),
        ("early_exit", ctypes.c_int32),
        ("schedule", ctypes.c_int32),
        ("probe_interval", ctypes.c_int32),
        ("cool_steps", ctypes.c_int32),
        ("gate_state", ctypes.c_void_p),
        ("step_dev", ctypes.c_void_p),
    ]


class KvPoolC(ctypes.Structure):
    _fields_ = [
        ("free_stack", ctypes.c_void_p),
        ("free_top", ctypes.c_void_p),
        ("block_table", ctypes.c_void_p),
        ("nblocks", ctypes.c_void_p),
        ("num_blocks", ctypes.c_int32),
        ("B", ctypes.c_int32),
        ("max_blocks", ctypes.c_int32),
        ("block_size", ctypes.c_int32),
    ]


SCHEDULE_AUTO, SCHEDULE_FUSED, SCHEDULE_SPLIT = 0, 1, 2


@dataclass
class VerifyParams:
    """Scalar knobs of spec_verify (see specng_verify_params)."""
    temperature: float = 1.0
    softcap: float = 0.0
    rep_penalty: float = 1.0
    rep_window: int = 0
    ema_tau: float = 0.1
    ema_thresh: float = 0.5
    gate_enabled: bool = True
    seed: int = 0
    step: int = 0
    early_exit: bool = False      # skip the rows past a known first rejection (same outputs)
    schedule: int = SCHEDULE_AUTO
    probe_interval: int = 0       # gate variant: re-probe a gated-off sequence every this many steps
    cool_steps: int = 0           # gate variant: no drafts for this many calls after a partial acceptance
    gate_state: Optional[torch.Tensor] = None  # int32 [B] cooling counts (in/out), needed with cool_steps
    step_dev: Optional[torch.Tensor] = None    # int64 [1] device step counter (read instead of step)

    def to_c(self) -> VerifyParamsC:
        gs = None
        if self.gate_state is not None:
            gs = _ptr(self.gate_state, torch.int32, "gate_state").value
        sd = None
        if self.step_dev is not None:
            sd = _ptr(self.step_dev, torch.int64, "step_dev").value
        return VerifyParamsC(self.temperature, self.softcap, self.rep_penalty, int(self.rep_window),
                             self.ema_tau, self.ema_thresh, 1 if self.gate_enabled else 0, 0,
                             int(self.seed) & 0xFFFFFFFFFFFFFFFF, int(self.step) & 0xFFFFFFFFFFFFFFFF,
                             1 if self.early_exit else 0, int(self.schedule), int(self.probe_interval),
                             int(self.cool_steps), gs, sd)


_lib = None


def lib_path() -> str:
    return _LIB_PATH


def load() -> ctypes.CDLL:
    """Load libspecng.so (built by ``build()``); raises if it is absent."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(_LIB_PATH):
        raise SpecngError(f"{_LIB_PATH} is missing: build the CUDA library first "
                          "(python -m speculative_decoding_draft_ngram_gb300.build)")
    L = ctypes.CDLL(_LIB_PATH)
    P, I, I64, SZ, U64 = ctypes.c_void_p, ctypes.c_int, ctypes.c_int64, ctypes.c_size_t, ctypes.c_uint64
    sig = {
        "specng_ngram_create": (I, [ctypes.POINTER(P), I, I, I64, P]),
        "specng_ngram_destroy": (I, [P]),
        "specng_ngram_reset": (I, [P, P]),
        "specng_ngram_capacity": (I, [P, ctypes.POINTER(I64)]),
        "specng_ngram_set_min_count": (I, [P, I]),
        "ngram_update": (I, [P, I64, P, P, P]),
        "ngram_draft": (I, [P, P, I64, P, I, P, P, P, P, P]),
        "spec_verify_workspace_bytes": (SZ, [I, I, I]),
        "spec_verify_workspace_init": (I, [P, SZ, P]),
        "spec_verify": (I, [P, I, I, I, I, P, P, P, P, I64, P, ctypes.POINTER(VerifyParamsC),
                            P, P, P, P, P, SZ, P]),
        "spec_verify_noalloc": (I, [P, I, I, I, I, P, P, P, P, I64, P, ctypes.POINTER(VerifyParamsC),
                                    P, P, P, P, P]),
        "spec_verify_lmhead_workspace_bytes": (SZ, [I, I, I]),
        "spec_verify_lmhead": (I, [P, P, I, P, I, I, I, P, P, P, P, I64, P, ctypes.POINTER(VerifyParamsC),
                                   P, P, P, P, P, SZ, P]),
        "spec_append": (I, [P, I64, P, I64, P, P, I, I, P]),
        "spec_commit": (I, [P, P, I64, P, I64, P, P, I, I, I, P, P, P, P, P]),
        "specng_get_status": (I, [ctypes.POINTER(ctypes.c_uint32), I]),
        "specng_get_counters": (I, [ctypes.POINTER(ctypes.c_uint32), I, I]),
        "specng_set_verify_marker": (I, [P]),
        "specng_strerror": (ctypes.c_char_p, [I]),
        "specng_last_error": (ctypes.c_char_p, []),
        "specng_philox4x32_10": (I, [P, U64, P, I64, P]),
        "specng_kv_init": (I, [ctypes.POINTER(KvPoolC), P]),
        "specng_kv_reserve": (I, [ctypes.POINTER(KvPoolC), P, I, P]),
        "specng_kv_trim": (I, [ctypes.POINTER(KvPoolC), P, P]),
        "specng_kv_release": (I, [ctypes.POINTER(KvPoolC), P, P]),
        "specng_step_advance": (I, [P, P]),
    }
    for name, (res, args) in sig.items():
        f = getattr(L, name)
        f.restype = res
        f.argtypes = args
    _lib = L
    return L


def _check(rc: int, what: str):
    if rc != SPECNG_OK:
        L = load()
        raise SpecngError(f"{what} failed ({rc}: {L.specng_strerror(rc).decode()}): "
                          f"{L.specng_last_error().decode()}")


def _ptr(t: Optional[torch.Tensor], dtype=None, name="tensor"):
    if t is None:
        return None
    if not t.is_cuda:
        raise SpecngError(f"{name} must be a CUDA tensor")
    if not t.is_contiguous():
        raise SpecngError(f"{name} must be contiguous")
    if dtype is not None and t.dtype != dtype:
        raise SpecngError(f"{name} must be {dtype}, got {t.dtype}")
    return ctypes.c_void_p(t.data_ptr())


def _stream(device=None):
    return ctypes.c_void_p(torch.cuda.current_stream(device).cuda_stream)


# ---------------------------------------------------------------- n-gram

class NgramTable:
    """Device n-gram table (owns its memory; see specng_ngram_create)."""

    def __init__(self, B: int, V: int, max_positions: int, device=None):
        L = load()
        self.B, self.V = int(B), int(V)
        self.device = torch.device(device if device is not None else "cuda")
        self._h = ctypes.c_void_p()
        with torch.cuda.device(self.device):
            _check(L.specng_ngram_create(ctypes.byref(self._h), self.B, self.V, int(max_positions),
                                         _stream(self.device)), "specng_ngram_create")

    @property
    def capacity(self) -> int:
        n = ctypes.c_int64()
        _check(load().specng_ngram_capacity(self._h, ctypes.byref(n)), "specng_ngram_capacity")
        return n.value

    def reset(self):
        _check(load().specng_ngram_reset(self._h, _stream(self.device)), "specng_ngram_reset")

    def set_min_count(self, min_count: int):
        """Draft only continuations seen at least min_count times (1: any)."""
        _check(load().specng_ngram_set_min_count(self._h, int(min_count)), "specng_ngram_set_min_count")

    def close(self):
        if self._h is not None and self._h.value:
            with torch.cuda.device(self.device):
                _check(load().specng_ngram_destroy(self._h), "specng_ngram_destroy")
        self._h = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass


def ngram_update(table: NgramTable, history: torch.Tensor, lens: torch.Tensor):
    """Index positions [indexed_b, lens_b) of every sequence (two kernels)."""
    with torch.cuda.device(history.device):
        _check(load().ngram_update(_ptr(history, torch.int32, "history"), history.shape[1],
                                   _ptr(lens, torch.int32, "lens"), table._h, _stream(history.device)),
               "ngram_update")


def ngram_draft(table: NgramTable, history: torch.Tensor, lens: torch.Tensor, max_k: int,
                k_limit: Optional[torch.Tensor] = None, out_drafts: Optional[torch.Tensor] = None,
                out_k: Optional[torch.Tensor] = None, fallback: Optional[torch.Tensor] = None):
    """Chained trigram -> bigram drafts: returns (out_drafts [B, max_k], out_k [B]).

    fallback [B, max_k] (optional) fills the positions after the first miss."""
    B = lens.shape[0]
    if out_drafts is None:
        out_drafts = torch.empty((B, max_k), dtype=torch.int32, device=history.device)
    if out_k is None:
        out_k = torch.empty((B,), dtype=torch.int32, device=history.device)
    with torch.cuda.device(history.device):
        _check(load().ngram_draft(table._h, _ptr(history, torch.int32, "history"), history.shape[1],
                                  _ptr(lens, torch.int32, "lens"), int(max_k),
                                  _ptr(k_limit, torch.int32, "k_limit"), _ptr(fallback, torch.int32, "fallback"),
                                  _ptr(out_drafts, torch.int32, "out_drafts"),
                                  _ptr(out_k, torch.int32, "out_k"), _stream(history.device)), "ngram_draft")
    return out_drafts, out_k


# ---------------------------------------------------------------- verify

def spec_verify_workspace_bytes(B: int, K: int, V: int) -> int:
    return int(load().spec_verify_workspace_bytes(int(B), int(K), int(V)))


def spec_verify_workspace(B: int, K: int, V: int, device=None) -> torch.Tensor:
    """A zero-filled workspace tensor for spec_verify (allocated once, reused)."""
    n = spec_verify_workspace_bytes(B, K, V)
    return torch.zeros(n, dtype=torch.uint8, device=device if device is not None else "cuda")


def spec_verify(logits: torch.Tensor, drafts: Optional[torch.Tensor], draft_probs: Optional[torch.Tensor],
                k: torch.Tensor, history: Optional[torch.Tensor], lens: Optional[torch.Tensor],
                params: VerifyParams, kv_len: torch.Tensor, ema: torch.Tensor, out_tokens: torch.Tensor,
                out_accept_len: torch.Tensor, workspace: torch.Tensor):
    """One verify call; writes out_tokens / out_accept_len and updates kv_len / ema in place."""
    if logits.dim() != 3:
        raise SpecngError("logits must be [B, K+1, V]")
    B, K1, V = logits.shape
    if logits.dtype == torch.bfloat16:
        dt = SPECNG_BF16
    elif logits.dtype == torch.float32:
        dt = SPECNG_F32
    else:
        raise SpecngError(f"logits dtype {logits.dtype} unsupported (bfloat16 or float32)")
    pc = params.to_c()
    with torch.cuda.device(logits.device):   # the library works on the current device
        _check(load().spec_verify(
            _ptr(logits, None, "logits"), dt, B, K1 - 1, V,
            _ptr(drafts, torch.int32, "drafts"), _ptr(draft_probs, torch.float32, "draft_probs"),
            _ptr(k, torch.int32, "k"), _ptr(history, torch.int32, "history"),
            history.shape[1] if history is not None else 0, _ptr(lens, torch.int32, "lens"),
            ctypes.byref(pc), _ptr(kv_len, torch.int32, "kv_len"), _ptr(ema, torch.float32, "ema"),
            _ptr(out_tokens, torch.int32, "out_tokens"), _ptr(out_accept_len, torch.int32, "out_accept_len"),
            _ptr(workspace, None, "workspace"), workspace.numel() * workspace.element_size(),
            _stream(logits.device)), "spec_verify")


def spec_verify_noalloc(logits: torch.Tensor, drafts: Optional[torch.Tensor], draft_probs: Optional[torch.Tensor],
                        k: torch.Tensor, history: Optional[torch.Tensor], lens: Optional[torch.Tensor],
                        params: VerifyParams, kv_len: torch.Tensor, ema: torch.Tensor, out_tokens: torch.Tensor,
                        out_accept_len: torch.Tensor):
    """spec_verify on the library's static scratch (no workspace, nothing allocated).

    For callers that cannot allocate device memory where they verify; shapes
    are limited to spec_verify_workspace_bytes(B, K, V) <= 16 MiB, and calls
    on one device must not overlap (they share the scratch)."""
    if logits.dim() != 3:
        raise SpecngError("logits must be [B, K+1, V]")
    B, K1, V = logits.shape
    if logits.dtype == torch.bfloat16:
        dt = SPECNG_BF16
    elif logits.dtype == torch.float32:
        dt = SPECNG_F32
    else:
        raise SpecngError(f"logits dtype {logits.dtype} unsupported (bfloat16 or float32)")
    pc = params.to_c()
    with torch.cuda.device(logits.device):   # the scratch is the current device's
        _check(load().spec_verify_noalloc(
            _ptr(logits, None, "logits"), dt, B, K1 - 1, V,
            _ptr(drafts, torch.int32, "drafts"), _ptr(draft_probs, torch.float32, "draft_probs"),
            _ptr(k, torch.int32, "k"), _ptr(history, torch.int32, "history"),
            history.shape[1] if history is not None else 0, _ptr(lens, torch.int32, "lens"),
            ctypes.byref(pc), _ptr(kv_len, torch.int32, "kv_len"), _ptr(ema, torch.float32, "ema"),
            _ptr(out_tokens, torch.int32, "out_tokens"), _ptr(out_accept_len, torch.int32, "out_accept_len"),
            _stream(logits.device)), "spec_verify_noalloc")


def spec_verify_lmhead_workspace_bytes(B: int, K: int, V: int) -> int:
    return int(load().spec_verify_lmhead_workspace_bytes(int(B), int(K), int(V)))


def spec_verify_lmhead_workspace(B: int, K: int, V: int, device=None) -> torch.Tensor:
    """A zero-filled workspace tensor for spec_verify_lmhead (allocated once, reused)."""
    n = spec_verify_lmhead_workspace_bytes(B, K, V)
    return torch.zeros(n, dtype=torch.uint8, device=device if device is not None else "cuda")


def spec_verify_lmhead(hidden: torch.Tensor, weight: torch.Tensor, logits: torch.Tensor,
                       drafts: Optional[torch.Tensor], draft_probs: Optional[torch.Tensor], k: torch.Tensor,
                       history: Optional[torch.Tensor], lens: Optional[torch.Tensor], params: VerifyParams,
                       kv_len: torch.Tensor, ema: torch.Tensor, out_tokens: torch.Tensor,
                       out_accept_len: torch.Tensor, workspace: torch.Tensor):
    """Fused LM head + verify: logits = hidden weight^T (written, bf16) and the verify of the drafts.

    hidden [B, K+1, d] bf16, weight [V, d] bf16, logits [B, K+1, V] bf16 (output)."""
    if hidden.dim() != 3 or weight.dim() != 2 or logits.dim() != 3:
        raise SpecngError("hidden must be [B, K+1, d], weight [V, d], logits [B, K+1, V]")
    B, K1, d = hidden.shape
    V = weight.shape[0]
    if weight.shape[1] != d or tuple(logits.shape) != (B, K1, V):
        raise SpecngError("shapes of hidden, weight and logits disagree")
    for name, t in (("hidden", hidden), ("weight", weight), ("logits", logits)):
        if t.dtype != torch.bfloat16:
            raise SpecngError(f"{name} must be bfloat16")
    pc = params.to_c()
    with torch.cuda.device(logits.device):   # the library works on the current device
        _check(load().spec_verify_lmhead(
            _ptr(hidden, None, "hidden"), _ptr(weight, None, "weight"), d, _ptr(logits, None, "logits"),
            B, K1 - 1, V,
            _ptr(drafts, torch.int32, "drafts"), _ptr(draft_probs, torch.float32, "draft_probs"),
            _ptr(k, torch.int32, "k"), _ptr(history, torch.int32, "history"),
            history.shape[1] if history is not None else 0, _ptr(lens, torch.int32, "lens"),
            ctypes.byref(pc), _ptr(kv_len, torch.int32, "kv_len"), _ptr(ema, torch.float32, "ema"),
            _ptr(out_tokens, torch.int32, "out_tokens"), _ptr(out_accept_len, torch.int32, "out_accept_len"),
            _ptr(workspace, None, "workspace"), workspace.numel() * workspace.element_size(),
            _stream(logits.device)), "spec_verify_lmhead")


def spec_append(history: torch.Tensor, lens: torch.Tensor, out_tokens: torch.Tensor,
                out_accept_len: torch.Tensor, hist_cap: Optional[int] = None):
    """history[b, lens_b + t] = out_tokens[b, t] for t <= a_b; lens_b += a_b + 1 (in place)."""
    B, K1 = out_tokens.shape
    cap = history.shape[1] if hist_cap is None else int(hist_cap)
    with torch.cuda.device(history.device):
        _check(load().spec_append(_ptr(history, torch.int32, "history"), history.shape[1],
                                  _ptr(lens, torch.int32, "lens"), cap, _ptr(out_tokens, torch.int32, "out_tokens"),
                                  _ptr(out_accept_len, torch.int32, "out_accept_len"), B, K1 - 1,
                                  _stream(history.device)), "spec_append")


def spec_commit(table: NgramTable, history: torch.Tensor, lens: torch.Tensor, out_tokens: torch.Tensor,
                out_accept_len: torch.Tensor, max_k: int, k_limit: Optional[torch.Tensor] = None,
                fallback: Optional[torch.Tensor] = None, out_drafts: Optional[torch.Tensor] = None,
                out_k: Optional[torch.Tensor] = None, hist_cap: Optional[int] = None):
    """spec_append + ngram_update + ngram_draft (next step) in one launch;
    returns (out_drafts [B, max_k], out_k [B])."""
    B, K1 = out_tokens.shape
    if out_drafts is None:
        out_drafts = torch.empty((B, max_k), dtype=torch.int32, device=history.device)
    if out_k is None:
        out_k = torch.empty((B,), dtype=torch.int32, device=history.device)
    cap = history.shape[1] if hist_cap is None else int(hist_cap)
    with torch.cuda.device(history.device):
        _check(load().spec_commit(table._h, _ptr(history, torch.int32, "history"), history.shape[1],
                                  _ptr(lens, torch.int32, "lens"), cap, _ptr(out_tokens, torch.int32, "out_tokens"),
                                  _ptr(out_accept_len, torch.int32, "out_accept_len"), B, K1 - 1, int(max_k),
                                  _ptr(k_limit, torch.int32, "k_limit"), _ptr(fallback, torch.int32, "fallback"),
                                  _ptr(out_drafts, torch.int32, "out_drafts"), _ptr(out_k, torch.int32, "out_k"),
                                  _stream(history.device)), "spec_commit")
    return out_drafts, out_k


# ---------------------------------------------------------------- decode-step bookkeeping

class KvPool:
    """Bookkeeping of a pool of KV blocks (see specng_kv_pool): the free-block
    stack and the per-sequence block tables, as int32 device tensors."""

    def __init__(self, num_blocks: int, B: int, max_blocks: int, block_size: int, device=None):
        self.device = torch.device(device if device is not None else "cuda")
        self.num_blocks, self.B = int(num_blocks), int(B)
        self.max_blocks, self.block_size = int(max_blocks), int(block_size)
        self.free_stack = torch.empty(self.num_blocks, dtype=torch.int32, device=self.device)
        self.free_top = torch.empty(1, dtype=torch.int32, device=self.device)
        self.block_table = torch.empty((self.B, self.max_blocks), dtype=torch.int32, device=self.device)
        self.nblocks = torch.empty(self.B, dtype=torch.int32, device=self.device)
        self.init()

    def _c(self) -> KvPoolC:
        return KvPoolC(self.free_stack.data_ptr(), self.free_top.data_ptr(), self.block_table.data_ptr(),
                       self.nblocks.data_ptr(), self.num_blocks, self.B, self.max_blocks, self.block_size)

    def init(self):
        c = self._c()
        with torch.cuda.device(self.device):
            _check(load().specng_kv_init(ctypes.byref(c), _stream(self.device)), "specng_kv_init")

    def reserve(self, kv_len: torch.Tensor, extra: int):
        c = self._c()
        with torch.cuda.device(self.device):
            _check(load().specng_kv_reserve(ctypes.byref(c), _ptr(kv_len, torch.int32, "kv_len"), int(extra),
                                            _stream(self.device)), "specng_kv_reserve")

    def trim(self, kv_len: torch.Tensor):
        c = self._c()
        with torch.cuda.device(self.device):
            _check(load().specng_kv_trim(ctypes.byref(c), _ptr(kv_len, torch.int32, "kv_len"),
                                         _stream(self.device)), "specng_kv_trim")

    def release(self, done: torch.Tensor):
        c = self._c()
        with torch.cuda.device(self.device):
            _check(load().specng_kv_release(ctypes.byref(c), _ptr(done, torch.int32, "done"),
                                            _stream(self.device)), "specng_kv_release")


def step_advance(step_dev: torch.Tensor):
    """step_dev += 1 on the current stream (int64 [1] device tensor)."""
    with torch.cuda.device(step_dev.device):
        _check(load().specng_step_advance(_ptr(step_dev, torch.int64, "step_dev"), _stream(step_dev.device)),
               "specng_step_advance")


# ---------------------------------------------------------------- diagnostics

def set_verify_marker(event: Optional["torch.cuda.Event"]):
    """Record `event` after the streaming kernel of every later spec_verify
    call (None: stop).  The event must already exist (recorded once)."""
    h = None if event is None else ctypes.c_void_p(event.cuda_event)
    _check(load().specng_set_verify_marker(h), "specng_set_verify_marker")


def get_counters(clear: bool = True) -> dict:
    """Diagnostic counters of the current device (synchronises): how often each
    exact (fp64) decision path ran since the last clear (see DIAG)."""
    v = (ctypes.c_uint32 * DIAG_N)()
    _check(load().specng_get_counters(v, DIAG_N, 1 if clear else 0), "specng_get_counters")
    return {name: int(v[i]) for name, i in DIAG.items()}


def get_status(clear: bool = True) -> int:
    """Device status bits (synchronises the device)."""
    v = ctypes.c_uint32()
    _check(load().specng_get_status(ctypes.byref(v), 1 if clear else 0), "specng_get_status")
    return v.value


def status_names(bits: int):
    return [n for b, n in STATUS_BITS.items() if bits & b]


def philox4x32_10(ctr: torch.Tensor, seed: int) -> torch.Tensor:
    """Philox4x32-10 of n counters (int32 tensor [n, 4] holding uint32 bits)."""
    out = torch.empty_like(ctr)
    _check(load().specng_philox4x32_10(_ptr(ctr, torch.int32, "ctr"), int(seed) & 0xFFFFFFFFFFFFFFFF,
                                       _ptr(out, torch.int32, "out"), ctr.shape[0], _stream(ctr.device)),
           "specng_philox4x32_10")
    return out
