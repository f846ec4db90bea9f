"""Thin ctypes binding of ``libspecverify.so`` (declared in include/specverify.h).

Argument marshalling only: every step of the verify path runs in the CUDA
library.  Functions take torch CUDA tensors (contiguous, on the current device)
and launch on the current torch stream unless ``stream`` is given.  There is no
CPU fallback: if the library is missing this module raises on first use.
"""
from __future__ import annotations

import ctypes
import os

import torch

HERE = os.path.dirname(os.path.abspath(__file__))
LIB = os.path.join(HERE, "libspecverify.so")

SV_OK, SV_ERR_INVALID_ARG, SV_ERR_WORKSPACE, SV_ERR_UNSUPPORTED, SV_ERR_CUDA, SV_ERR_DATA, \
    SV_ERR_TIMEOUT = range(7)
SV_BF16, SV_F32 = 0, 1
SV_MODE_SAMPLE, SV_MODE_GREEDY = 0, 1
SV_DEV_BAD_ROW, SV_DEV_BAD_TOKEN, SV_DEV_BAD_UNIFORM, SV_DEV_BAD_Q, SV_DEV_DEGENERATE = (
    0x1, 0x2, 0x4, 0x8, 0x10)
SV_DEV_PRECISE = 0x20
SV_DEV_BAD_TREE = 0x40

EXPORTS = ("spec_verify_workspace_size", "spec_verify_greedy", "spec_verify_sample",
           "spec_verify_rows", "spec_verify_finish", "spec_verify_read_status",
           "spec_verify_row_stats", "spec_verify_status_string", "spec_verify_sample_noalloc")
SV_NOALLOC_SCRATCH_BYTES = 1048576
SV_NOALLOC_MAX_ROWS = 27000

_lib = None


class Tuning(ctypes.Structure):
    """sv_tuning (specverify_debug.h): options of one call, for tests and tuning;
    every field 0 is the automatic choice.  Passed as ``tuning=`` to the wrappers
    below, it affects that call only."""
    _fields_ = [(name, ctypes.c_int) for name in (
        "path", "force_precise", "draw_split", "precise_split", "fused_defer",
        "fused_pad_kib", "rows_split", "rows_threads", "flat_off", "draw_mode")]


class SpecVerifyError(RuntimeError):
    def __init__(self, status: int, where: str):
        super().__init__(f"{where}: {status_string(status)} (status {status})")
        self.status = status


def load():
    """Load the CUDA library (raises if it has not been built)."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(LIB):
        raise ImportError(f"libspecverify.so is not built ({LIB}); run "
                          "speculative_decoding_verification_18_gb300.build.build() first")
    lib = ctypes.CDLL(LIB)
    P, I, F, Z = ctypes.c_void_p, ctypes.c_int, ctypes.c_float, ctypes.c_size_t
    lib.spec_verify_workspace_size.argtypes = [I, I, I, I]
    lib.spec_verify_workspace_size.restype = Z
    lib.spec_verify_greedy.argtypes = [P, I, P, I, I, I, P, P, P, Z, P]
    lib.spec_verify_greedy.restype = I
    lib.spec_verify_sample.argtypes = [P, I, P, P, P, P, F, I, I, I, P, P, P, Z, P]
    lib.spec_ngram_draft.argtypes = [P, P, I, I, I, I, I, P, P, P]
    lib.spec_ngram_draft.restype = I
    lib.spec_verify_match.argtypes = [P, I, P, P, P, F, I, I, I, P, P, P, Z, P]
    lib.spec_verify_match.restype = I
    lib.spec_verify_tree.argtypes = [I, P, I, P, P, P, P, P, F, I, I, I, P, P, P, P, Z, P]
    lib.spec_verify_tree.restype = I
    lib.spec_verify_sample_kv.argtypes = [P, I, P, P, P, P, F, I, I, I, P, P, P, Z, P, P, P]
    lib.spec_verify_sample_kv.restype = I
    lib.spec_verify_greedy_kv.argtypes = [P, I, P, I, I, I, P, P, P, Z, P, P, P]
    lib.spec_verify_greedy_kv.restype = I
    lib.spec_verify_sample.restype = I
    lib.spec_verify_rows.argtypes = [I, P, I, P, P, F, I, I, I, P, Z, P]
    lib.spec_verify_rows.restype = I
    lib.spec_verify_finish.argtypes = [I, P, I, P, P, P, P, F, I, I, I, P, P, P, Z, P]
    lib.spec_verify_finish.restype = I
    lib.spec_verify_debug_flat_ctas.argtypes = [I, I, I, I]
    lib.spec_verify_debug_flat_ctas.restype = I
    lib.spec_verify_sample_tuned.argtypes = [P, I, P, P, P, P, F, I, I, I, P, P, P, Z, P, P, P, P]
    lib.spec_verify_sample_tuned.restype = I
    lib.spec_verify_greedy_tuned.argtypes = [P, I, P, I, I, I, P, P, P, Z, P, P, P, P]
    lib.spec_verify_greedy_tuned.restype = I
    lib.spec_verify_rows_tuned.argtypes = [I, P, I, P, P, F, I, I, I, P, Z, P, P]
    lib.spec_verify_rows_tuned.restype = I
    lib.spec_verify_finish_tuned.argtypes = [I, P, I, P, P, P, P, F, I, I, I, P, P, P, Z, P, P]
    lib.spec_verify_finish_tuned.restype = I
    lib.spec_verify_tree_tuned.argtypes = [I, P, I, P, P, P, P, P, F, I, I, I, P, P, P, P, Z, P, P]
    lib.spec_verify_tree_tuned.restype = I
    lib.spec_verify_match_tuned.argtypes = [P, I, P, P, P, F, I, I, I, P, P, P, Z, P, P]
    lib.spec_verify_match_tuned.restype = I
    lib.spec_verify_debug_rows_skip.argtypes = [I, P, I, P, P, P, F, I, I, I, P, Z, P]
    lib.spec_verify_debug_rows_skip.restype = I
    lib.spec_verify_read_status.argtypes = [P, P, P, P]
    lib.spec_verify_read_status.restype = I
    lib.spec_verify_row_stats.argtypes = [P, P, I, I, P, P, P, P, P]
    lib.spec_verify_row_stats.restype = I
    lib.spec_verify_status_string.argtypes = [I]
    lib.spec_verify_status_string.restype = ctypes.c_char_p
    lib.spec_verify_sample_noalloc.argtypes = [P, I, P, P, P, P, F, I, I, I, P, P, P]
    lib.spec_verify_sample_noalloc.restype = I
    lib.spec_verify_debug_ffexp.argtypes = [P, F, F, I, P, P]
    lib.spec_verify_debug_ffexp.restype = I
    lib.spec_verify_debug_path.argtypes = [I, I, I, I]
    lib.spec_verify_debug_path.restype = I
    lib.spec_verify_debug_status_counts.argtypes = [P, P, P]
    lib.spec_verify_debug_status_counts.restype = I
    lib.spec_verify_debug_ex2_error.argtypes = [F, F, P, P]
    lib.spec_verify_debug_ex2_error.restype = I
    _lib = lib
    return lib


def status_string(status: int) -> str:
    return load().spec_verify_status_string(int(status)).decode()


def _ptr(t):
    if t is None:
        return None
    if isinstance(t, int):
        return t
    if not t.is_contiguous():
        raise ValueError("tensors must be contiguous")
    return t.data_ptr()


def _stream(stream):
    if stream is None:
        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, int):
        return stream
    return stream.cuda_stream


def _dtype(logits):
    if logits.dtype == torch.bfloat16:
        return SV_BF16
    if logits.dtype == torch.float32:
        return SV_F32
    raise TypeError(f"logits must be bfloat16 or float32, not {logits.dtype}")


def _check(st, where):
    if st != SV_OK:
        raise SpecVerifyError(st, where)


def spec_verify_workspace_size(B: int, k: int, V: int, dtype=SV_BF16) -> int:
    return int(load().spec_verify_workspace_size(B, k, V, dtype))


def _tun(tuning):
    return None if tuning is None else ctypes.byref(tuning)


def spec_verify_greedy(logits, draft_tokens, out_tokens, num_accepted, ws, stream=None,
                       tuning=None):
    """logits [B,k+1,V] bf16/fp32, draft_tokens [B,k] int32 -> out_tokens [B,k+1], num_accepted [B]."""
    B, k1, V = logits.shape
    args = (_ptr(logits), _dtype(logits), _ptr(draft_tokens), B, k1 - 1, V, _ptr(out_tokens),
            _ptr(num_accepted), _ptr(ws), ws.numel())
    if tuning is None:
        st = load().spec_verify_greedy(*args, _stream(stream))
    else:
        st = load().spec_verify_greedy_tuned(*args, None, None, _stream(stream), _tun(tuning))
    _check(st, "spec_verify_greedy")


def spec_verify_sample(logits, draft_probs, draft_tokens, u_accept, u_resample, T, out_tokens,
                       num_accepted, ws, stream=None, tuning=None):
    B, k1, V = logits.shape
    args = (_ptr(logits), _dtype(logits), _ptr(draft_probs), _ptr(draft_tokens), _ptr(u_accept),
            _ptr(u_resample), float(T), B, k1 - 1, V, _ptr(out_tokens), _ptr(num_accepted),
            _ptr(ws), ws.numel())
    if tuning is None:
        st = load().spec_verify_sample(*args, _stream(stream))
    else:
        st = load().spec_verify_sample_tuned(*args, None, None, _stream(stream), _tun(tuning))
    _check(st, "spec_verify_sample")


def spec_verify_match(logits, draft_tokens, u_draw, u_bonus, T, out_tokens, num_accepted, ws,
                      stream=None, tuning=None):
    """Sample-and-match verify: a target draw per position, drafts kept while equal."""
    B, k1, V = logits.shape
    args = (_ptr(logits), _dtype(logits), _ptr(draft_tokens), _ptr(u_draw), _ptr(u_bonus),
            float(T), B, k1 - 1, V, _ptr(out_tokens), _ptr(num_accepted), _ptr(ws), ws.numel(),
            _stream(stream))
    if tuning is None:
        st = load().spec_verify_match(*args)
    else:
        st = load().spec_verify_match_tuned(*args, _tun(tuning))
    _check(st, "spec_verify_match")


def spec_verify_tree(mode, logits, draft_probs, tree_tokens, tree_parents, u_accept, u_resample,
                     T, out_tokens, out_nodes, num_accepted, ws, stream=None, tuning=None):
    """Tree verify: logits [B, N, V], draft_probs [B, N, V] (sampled), tree_tokens and
    tree_parents [B, N] int32, u_accept [B, N], u_resample [B] -> out_tokens,
    out_nodes [B, N], num_accepted [B].  Workspace: workspace(B, N - 1, V, ...)."""
    B, N, V = logits.shape
    args = (int(mode), _ptr(logits), _dtype(logits), _ptr(draft_probs), _ptr(tree_tokens),
            _ptr(tree_parents), _ptr(u_accept), _ptr(u_resample), float(T), B, N, V,
            _ptr(out_tokens), _ptr(out_nodes), _ptr(num_accepted), _ptr(ws), ws.numel(),
            _stream(stream))
    if tuning is None:
        st = load().spec_verify_tree(*args)
    else:
        st = load().spec_verify_tree_tuned(*args, _tun(tuning))
    _check(st, "spec_verify_tree")


def spec_ngram_draft(history, lengths, k, n_min, n_max, draft_tokens, num_drafted, stream=None):
    """N-gram drafter: history [B, Lmax] int32, lengths [B] int32 -> draft_tokens [B, k],
    num_drafted [B]."""
    B, Lmax = history.shape
    st = load().spec_ngram_draft(_ptr(history), _ptr(lengths), B, Lmax, int(k), int(n_min),
                                 int(n_max), _ptr(draft_tokens), _ptr(num_drafted),
                                 _stream(stream))
    _check(st, "spec_ngram_draft")


STATS_FIELDS = ("rounds", "proposed", "accepted", "emitted", "invalid")


def stats_tensor(device=None):
    """Zeroed device counters laid out as sv_spec_stats (int64[5], 16-byte aligned)."""
    return torch.zeros(len(STATS_FIELDS), dtype=torch.int64, device=device or "cuda")


def stats_dict(stats):
    """sv_spec_stats counters (a stats_tensor) as a dict of ints."""
    v = stats.cpu().tolist()
    return dict(zip(STATS_FIELDS, (int(x) for x in v)))


def spec_verify_sample_kv(logits, draft_probs, draft_tokens, u_accept, u_resample, T, out_tokens,
                          num_accepted, ws, kv_len=None, stats=None, stream=None, tuning=None):
    """spec_verify_sample, then kv_len[b] += n + 1 and the stats counters, in the kernel."""
    B, k1, V = logits.shape
    args = (_ptr(logits), _dtype(logits), _ptr(draft_probs), _ptr(draft_tokens), _ptr(u_accept),
            _ptr(u_resample), float(T), B, k1 - 1, V, _ptr(out_tokens), _ptr(num_accepted),
            _ptr(ws), ws.numel(), _ptr(kv_len), _ptr(stats), _stream(stream))
    if tuning is None:
        st = load().spec_verify_sample_kv(*args)
    else:
        st = load().spec_verify_sample_tuned(*args, _tun(tuning))
    _check(st, "spec_verify_sample_kv")


def spec_verify_greedy_kv(logits, draft_tokens, out_tokens, num_accepted, ws, kv_len=None,
                          stats=None, stream=None, tuning=None):
    """spec_verify_greedy, then kv_len[b] += n + 1 and the stats counters, in the kernel."""
    B, k1, V = logits.shape
    args = (_ptr(logits), _dtype(logits), _ptr(draft_tokens), B, k1 - 1, V, _ptr(out_tokens),
            _ptr(num_accepted), _ptr(ws), ws.numel(), _ptr(kv_len), _ptr(stats), _stream(stream))
    if tuning is None:
        st = load().spec_verify_greedy_kv(*args)
    else:
        st = load().spec_verify_greedy_tuned(*args, _tun(tuning))
    _check(st, "spec_verify_greedy_kv")


def spec_verify_sample_noalloc(logits, draft_probs, draft_tokens, u_accept, u_resample, T,
                               out_tokens, num_accepted, stream=None):
    """spec_verify_sample without a workspace: scratch lives in a fixed device array
    of the library (B*(k+1) <= SV_NOALLOC_MAX_ROWS)."""
    B, k1, V = logits.shape
    st = load().spec_verify_sample_noalloc(_ptr(logits), _dtype(logits), _ptr(draft_probs),
                                           _ptr(draft_tokens), _ptr(u_accept), _ptr(u_resample),
                                           float(T), B, k1 - 1, V, _ptr(out_tokens),
                                           _ptr(num_accepted), _stream(stream))
    _check(st, "spec_verify_sample_noalloc")


def spec_verify_rows(mode, logits, draft_probs, draft_tokens, T, ws, stream=None, tuning=None):
    B, k1, V = logits.shape
    args = (int(mode), _ptr(logits), _dtype(logits), _ptr(draft_probs), _ptr(draft_tokens),
            float(T), B, k1 - 1, V, _ptr(ws), ws.numel(), _stream(stream))
    if tuning is None:
        st = load().spec_verify_rows(*args)
    else:
        st = load().spec_verify_rows_tuned(*args, _tun(tuning))
    _check(st, "spec_verify_rows")


def debug_flat_ctas(B: int, k: int, V: int, dtype) -> int:
    """CTAs of the flat greedy row stream for these sizes (0: the per-row stream)."""
    dt = SV_BF16 if dtype in (torch.bfloat16, "bf16") else SV_F32
    r = load().spec_verify_debug_flat_ctas(int(B), int(k), int(V), dt)
    if r < 0:
        raise SpecVerifyError(SV_ERR_CUDA, "spec_verify_debug_flat_ctas")
    return r


def debug_rows_skip(mode, logits, draft_probs, draft_tokens, u_accept, T, ws, stream=None):
    """Timing hook: the row-skipping path's first stage (stop reset + row stream)."""
    B, k1, V = logits.shape
    st = load().spec_verify_debug_rows_skip(int(mode), _ptr(logits), _dtype(logits),
                                            _ptr(draft_probs), _ptr(draft_tokens), _ptr(u_accept),
                                            float(T), B, k1 - 1, V, _ptr(ws), ws.numel(),
                                            _stream(stream))
    _check(st, "spec_verify_debug_rows_skip")


def spec_verify_finish(mode, logits, draft_probs, draft_tokens, u_accept, u_resample, T,
                       out_tokens, num_accepted, ws, stream=None, tuning=None):
    B, k1, V = logits.shape
    args = (int(mode), _ptr(logits), _dtype(logits), _ptr(draft_probs), _ptr(draft_tokens),
            _ptr(u_accept), _ptr(u_resample), float(T), B, k1 - 1, V, _ptr(out_tokens),
            _ptr(num_accepted), _ptr(ws), ws.numel(), _stream(stream))
    if tuning is None:
        st = load().spec_verify_finish(*args)
    else:
        st = load().spec_verify_finish_tuned(*args, _tun(tuning))
    _check(st, "spec_verify_finish")


def spec_verify_read_status(ws, stream=None):
    """(status code, device status bits, number of zero-mass residual draws); syncs the stream."""
    bits = ctypes.c_uint32(0)
    ndeg = ctypes.c_uint32(0)
    st = load().spec_verify_read_status(_ptr(ws), _stream(stream), ctypes.byref(bits),
                                        ctypes.byref(ndeg))
    if st not in (SV_OK, SV_ERR_DATA):
        raise SpecVerifyError(st, "spec_verify_read_status")
    return st, int(bits.value), int(ndeg.value)


def spec_verify_row_stats(ws, B, k, stream=None):
    """Per-row statistics of the last call on ``ws`` as numpy arrays [B, k+1]."""
    import numpy as np
    R = B * (k + 1)
    m = np.zeros(R, np.float32)
    S = np.zeros(R, np.float32)
    am = np.zeros(R, np.int32)
    px = np.zeros(R, np.float32)
    qx = np.zeros(R, np.float32)
    c = lambda a: a.ctypes.data_as(ctypes.c_void_p)
    st = load().spec_verify_row_stats(_ptr(ws), _stream(stream), B, k, c(m), c(S), c(am), c(px),
                                      c(qx))
    _check(st, "spec_verify_row_stats")
    sh = (B, k + 1)
    return dict(m=m.reshape(sh), S=S.reshape(sh), argmax=am.reshape(sh), px=px.reshape(sh),
                qx=qx.reshape(sh))


def spec_verify_status_string(status: int) -> str:
    return status_string(status)


def debug_ffexp(l, m: float, T: float, stream=None):
    """exp((l - m)/T) by the draw's float-float exponential (test hook), as float64."""
    out = torch.empty(l.numel(), dtype=torch.float64, device=l.device)
    st = load().spec_verify_debug_ffexp(_ptr(l), float(m), float(T), l.numel(), _ptr(out),
                                        _stream(stream))
    _check(st, "spec_verify_debug_ffexp")
    return out


def debug_status_counts(ws, stream=None):
    """Per status bit (0..7), the number of sequences of the last call on ``ws``
    with it set; syncs the stream."""
    counts = (ctypes.c_uint32 * 8)()
    st = load().spec_verify_debug_status_counts(_ptr(ws), _stream(stream), counts)
    _check(st, "spec_verify_debug_status_counts")
    return [int(c) for c in counts]


PATH_TWO_KERNEL, PATH_FUSED, PATH_SKIP = 1, 2, 3


def debug_path(mode: int, B: int, V: int, dtype) -> int:
    """The path (PATH_*) the one-call entry points take for these sizes."""
    dt = SV_BF16 if dtype in (torch.bfloat16, "bf16") else SV_F32
    r = load().spec_verify_debug_path(int(mode), int(B), int(V), dt)
    if r < 0:
        raise SpecVerifyError(SV_ERR_CUDA, "spec_verify_debug_path")
    return r


def debug_ex2_error(a0: float, a1: float, stream=None) -> float:
    """Test hook: worst relative error of ex2.approx.ftz.f32 over every float in [a0, a1]."""
    out = torch.zeros(1, dtype=torch.float32, device="cuda")
    st = load().spec_verify_debug_ex2_error(float(a0), float(a1), _ptr(out), _stream(stream))
    _check(st, "spec_verify_debug_ex2_error")
    return float(out.item())


# ---------------------------------------------------------------- convenience

def workspace(B, k, V, dtype=torch.bfloat16, device=None):
    """A workspace tensor of the required size (bytes, uint8)."""
    n = spec_verify_workspace_size(B, k, V, SV_BF16 if dtype == torch.bfloat16 else SV_F32)
    return torch.empty(max(n, 256), dtype=torch.uint8, device=device or "cuda")


def verify_greedy(logits, draft_tokens, ws=None, stream=None):
    B, k1, V = logits.shape
    out = torch.empty((B, k1), dtype=torch.int32, device=logits.device)
    n = torch.empty(B, dtype=torch.int32, device=logits.device)
    if ws is None:
        ws = workspace(B, k1 - 1, V, logits.dtype, logits.device)
    spec_verify_greedy(logits, draft_tokens, out, n, ws, stream)
    return out, n


def verify_sample(logits, draft_probs, draft_tokens, u_accept, u_resample, T, ws=None,
                  stream=None):
    B, k1, V = logits.shape
    out = torch.empty((B, k1), dtype=torch.int32, device=logits.device)
    n = torch.empty(B, dtype=torch.int32, device=logits.device)
    if ws is None:
        ws = workspace(B, k1 - 1, V, logits.dtype, logits.device)
    spec_verify_sample(logits, draft_probs, draft_tokens, u_accept, u_resample, T, out, n, ws,
                       stream)
    return out, n
