"""ctypes binding of libspecverify (include/specverify.h).

Argument marshalling only: every step of the verify/sample computation runs in
the library's CUDA kernels.  The functions named like the C entry points take
raw integers (device addresses, sizes); ``verify_sample`` / ``verify_greedy``
take torch CUDA tensors, allocate the outputs and pass their addresses.
There is no fallback: if the library is missing or the tensors are not on a
CUDA device the call raises.
"""

from __future__ import annotations

import ctypes
import os

import torch

from .build import LIB_PATH

SV_OK = 0
SV_ERR_INVALID_ARG = 1
SV_ERR_UNSUPPORTED = 2
SV_ERR_WORKSPACE = 3
SV_ERR_CUDA = 4
SV_ERR_TIMEOUT = 5

SV_DTYPE_F32 = 0
SV_DTYPE_BF16 = 1
SV_DTYPE_F16 = 2

SV_SEQ_DRAFT_OUT_OF_RANGE = 1
SV_SEQ_Q_NOT_POSITIVE = 2
SV_SEQ_BAD_ROW = 4
SV_SEQ_RESIDUAL_ZERO = 8

# Size of the static scratch sv_verify_greedy_noalloc works in (the header's
# SV_NOALLOC_SCRATCH_BYTES).
SV_NOALLOC_SCRATCH_BYTES = 8 << 20

_TORCH_DTYPE = {torch.float32: SV_DTYPE_F32, torch.bfloat16: SV_DTYPE_BF16, torch.float16: SV_DTYPE_F16}

_c_int, _c_float, _c_size, _c_ptr = ctypes.c_int, ctypes.c_float, ctypes.c_size_t, ctypes.c_void_p

_lib = None


class SvError(RuntimeError):
    def __init__(self, status: int, what: str):
        super().__init__(f"{what}: {sv_status_string(status)}")
        self.status = status


def load_library(path: str = LIB_PATH) -> ctypes.CDLL:
    """Load libspecverify.so and declare its C signatures (raises if missing)."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(path):
        raise RuntimeError(f"{path} is missing: build it with "
                           "`python -c 'import __graft_entry__ as g; g.build()'`")
    lib = ctypes.CDLL(path)
    lib.sv_workspace_bytes.argtypes = [_c_int, _c_int, _c_int, _c_int]
    lib.sv_workspace_bytes.restype = _c_size
    lib.sv_verify_sample.argtypes = [_c_int, _c_int, _c_int, _c_ptr, _c_int, _c_ptr, _c_ptr, _c_ptr,
                                     _c_float, _c_int, _c_float, _c_ptr, _c_ptr, _c_ptr, _c_ptr,
                                     _c_ptr, _c_size, _c_ptr]
    lib.sv_verify_sample.restype = _c_int
    lib.sv_verify_greedy.argtypes = [_c_int, _c_int, _c_int, _c_ptr, _c_int, _c_ptr, _c_ptr, _c_ptr,
                                     _c_ptr, _c_ptr, _c_size, _c_ptr]
    lib.sv_verify_greedy.restype = _c_int
    lib.sv_status_string.argtypes = [_c_int]
    lib.sv_status_string.restype = ctypes.c_char_p
    lib.sv_verify_greedy_noalloc.argtypes = [_c_int, _c_int, _c_int, _c_ptr, _c_int, _c_ptr, _c_ptr, _c_ptr,
                                             _c_ptr, _c_ptr]
    lib.sv_verify_greedy_noalloc.restype = _c_int
    lib.sv_set_timing_events.argtypes = [ctypes.POINTER(_c_ptr), _c_int]
    lib.sv_set_timing_events.restype = _c_int
    lib.sv_verify_sample_ragged.argtypes = [_c_int, _c_int, _c_int, _c_ptr, _c_int, _c_ptr, _c_ptr, _c_ptr, _c_ptr,
                                            _c_float, _c_int, _c_float, _c_ptr, _c_ptr, _c_ptr, _c_ptr,
                                            _c_ptr, _c_size, _c_ptr]
    lib.sv_verify_sample_ragged.restype = _c_int
    lib.sv_verify_greedy_ragged.argtypes = [_c_int, _c_int, _c_int, _c_ptr, _c_int, _c_ptr, _c_ptr, _c_ptr, _c_ptr,
                                            _c_ptr, _c_ptr, _c_size, _c_ptr]
    lib.sv_verify_greedy_ragged.restype = _c_int
    lib.sv_truncate_emitted.argtypes = [_c_int, _c_int, _c_ptr, _c_ptr, _c_ptr, _c_int, _c_ptr, _c_ptr, _c_ptr]
    lib.sv_truncate_emitted.restype = _c_int
    lib.sv_last_kernels.argtypes = []
    lib.sv_last_kernels.restype = ctypes.c_char_p
    lib.sv_pointer_device_readable.argtypes = [_c_ptr]
    lib.sv_pointer_device_readable.restype = ctypes.c_int
    lib.sv_qlogits_workspace_bytes.argtypes = [_c_int, _c_int, _c_int, _c_int]
    lib.sv_qlogits_workspace_bytes.restype = _c_size
    lib.sv_verify_sample_qlogits.argtypes = [_c_int, _c_int, _c_int, _c_ptr, _c_int, _c_ptr, _c_int, _c_ptr, _c_ptr,
                                             _c_float, _c_int, _c_float, _c_ptr, _c_ptr, _c_ptr, _c_ptr,
                                             _c_ptr, _c_size, _c_ptr]
    lib.sv_verify_sample_qlogits.restype = _c_int
    lib.sv_shard_workspace_bytes.argtypes = [_c_int, _c_int, _c_int]
    lib.sv_shard_workspace_bytes.restype = _c_size
    lib.sv_shard_row_stats.argtypes = [_c_int, _c_int, _c_int, _c_int, _c_int, _c_ptr, _c_int, _c_ptr, _c_ptr,
                                       _c_float, _c_int, _c_ptr, _c_ptr]
    lib.sv_shard_row_stats.restype = _c_int
    lib.sv_shard_scan.argtypes = [_c_int, _c_int, _c_int, _c_int, _c_int, _c_ptr, _c_ptr, _c_ptr, _c_float, _c_int,
                                  _c_ptr, _c_ptr, _c_ptr, _c_ptr, _c_ptr, _c_size, _c_ptr]
    lib.sv_shard_scan.restype = _c_int
    lib.sv_shard_draw_sums.argtypes = [_c_int, _c_int, _c_int, _c_int, _c_int, _c_ptr, _c_int, _c_ptr, _c_ptr,
                                       _c_float, _c_ptr, _c_ptr, _c_size, _c_ptr]
    lib.sv_shard_draw_sums.restype = _c_int
    lib.sv_shard_draw_pick.argtypes = [_c_int, _c_int, _c_int, _c_int, _c_int, _c_int, _c_int, _c_ptr, _c_int,
                                       _c_ptr, _c_ptr, _c_ptr, _c_float, _c_ptr, _c_ptr, _c_ptr, _c_ptr, _c_size,
                                       _c_ptr]
    lib.sv_shard_draw_pick.restype = _c_int
    lib.sv_shard_topk_candidates.argtypes = [_c_int, _c_int, _c_int, _c_int, _c_int, _c_ptr, _c_int, _c_ptr, _c_ptr,
                                             _c_float, _c_int, _c_ptr, _c_ptr, _c_size, _c_ptr]
    lib.sv_shard_topk_candidates.restype = _c_int
    lib.sv_shard_topk_finish.argtypes = [_c_int, _c_int, _c_int, _c_int, _c_ptr, _c_ptr, _c_ptr, _c_float, _c_int,
                                         _c_float, _c_ptr, _c_ptr, _c_ptr, _c_ptr, _c_ptr]
    lib.sv_shard_topk_finish.restype = _c_int
    _lib = lib
    return lib


# ------------------------------------------------------------ raw C entry points

def sv_workspace_bytes(B: int, gamma: int, V: int, top_k: int = 0) -> int:
    return int(load_library().sv_workspace_bytes(B, gamma, V, top_k))


def sv_qlogits_workspace_bytes(B: int, gamma: int, V: int, top_k: int = 0) -> int:
    return int(load_library().sv_qlogits_workspace_bytes(B, gamma, V, top_k))


def sv_verify_sample_qlogits(B, gamma, V, logits, logits_dtype, q_logits, q_logits_dtype, draft_tokens, uniforms,
                             temperature, top_k, top_p, out_tokens, out_num_accepted, out_accept_prob, out_status,
                             workspace, workspace_bytes, stream) -> int:
    return int(load_library().sv_verify_sample_qlogits(B, gamma, V, logits, logits_dtype, q_logits, q_logits_dtype,
                                                        draft_tokens, uniforms, float(temperature), int(top_k),
                                                        float(top_p), out_tokens, out_num_accepted, out_accept_prob,
                                                        out_status, workspace, workspace_bytes, stream))


SV_MAX_SHARDS = 32
SV_SHARD_STAT_WORDS = 8
SV_SHARD_TOTAL_WORDS = 8


def sv_shard_workspace_bytes(B: int, gamma: int, V: int) -> int:
    return int(load_library().sv_shard_workspace_bytes(B, gamma, V))


def sv_shard_row_stats(B, gamma, V, v0, Vg, logits, logits_dtype, q, draft_tokens, temperature, greedy, stats_local,
                       stream) -> int:
    return int(load_library().sv_shard_row_stats(B, gamma, V, v0, Vg, logits, logits_dtype, q, draft_tokens,
                                                  float(temperature), int(greedy), stats_local, stream))


def sv_shard_scan(nshard, B, gamma, V, Vg, stats_all, draft_tokens, uniforms, temperature, greedy, out_tokens,
                  out_num_accepted, out_accept_prob, out_status, workspace, workspace_bytes, stream) -> int:
    return int(load_library().sv_shard_scan(nshard, B, gamma, V, Vg, stats_all, draft_tokens, uniforms,
                                             float(temperature), int(greedy), out_tokens, out_num_accepted,
                                             out_accept_prob, out_status, workspace, workspace_bytes, stream))


def sv_shard_draw_sums(B, gamma, V, v0, Vg, logits, logits_dtype, q, draft_tokens, temperature, totals_local,
                       workspace, workspace_bytes, stream) -> int:
    return int(load_library().sv_shard_draw_sums(B, gamma, V, v0, Vg, logits, logits_dtype, q, draft_tokens,
                                                  float(temperature), totals_local, workspace, workspace_bytes,
                                                  stream))


def sv_shard_draw_pick(nshard, rank, B, gamma, V, v0, Vg, logits, logits_dtype, q, draft_tokens, uniforms,
                       temperature, totals_all, out_tokens, out_status, workspace, workspace_bytes, stream) -> int:
    return int(load_library().sv_shard_draw_pick(nshard, rank, B, gamma, V, v0, Vg, logits, logits_dtype, q,
                                                  draft_tokens, uniforms, float(temperature), totals_all,
                                                  out_tokens, out_status, workspace, workspace_bytes, stream))


SV_SHARD_CAND_BYTES = 16


def sv_shard_topk_candidates(B, gamma, V, v0, Vg, logits, logits_dtype, q, draft_tokens, temperature, top_k,
                             cand_local, workspace, workspace_bytes, stream) -> int:
    return int(load_library().sv_shard_topk_candidates(B, gamma, V, v0, Vg, logits, logits_dtype, q, draft_tokens,
                                                        float(temperature), int(top_k), cand_local, workspace,
                                                        workspace_bytes, stream))


def sv_shard_topk_finish(nshard, B, gamma, Vg, cand_all, draft_tokens, uniforms, temperature, top_k, top_p,
                         out_tokens, out_num_accepted, out_accept_prob, out_status, stream) -> int:
    return int(load_library().sv_shard_topk_finish(nshard, B, gamma, Vg, cand_all, draft_tokens, uniforms,
                                                    float(temperature), int(top_k), float(top_p), out_tokens,
                                                    out_num_accepted, out_accept_prob, out_status, stream))


def sv_status_string(status: int) -> str:
    return load_library().sv_status_string(int(status)).decode()


def sv_verify_sample(B, gamma, V, logits, logits_dtype, q, draft_tokens, uniforms, temperature, top_k, top_p,
                     out_tokens, out_num_accepted, out_accept_prob, out_status, workspace, workspace_bytes,
                     stream) -> int:
    return int(load_library().sv_verify_sample(B, gamma, V, logits, logits_dtype, q, draft_tokens, uniforms,
                                                float(temperature), int(top_k), float(top_p), out_tokens,
                                                out_num_accepted, out_accept_prob, out_status, workspace,
                                                workspace_bytes, stream))


def sv_verify_greedy(B, gamma, V, logits, logits_dtype, draft_tokens, out_tokens, out_num_accepted, out_status,
                     workspace, workspace_bytes, stream) -> int:
    return int(load_library().sv_verify_greedy(B, gamma, V, logits, logits_dtype, draft_tokens, out_tokens,
                                               out_num_accepted, out_status, workspace, workspace_bytes, stream))


def sv_verify_greedy_noalloc(B, gamma, V, logits, logits_dtype, draft_tokens, out_tokens, out_num_accepted,
                             out_status, stream) -> int:
    """Greedy verify on the library's own scratch (no workspace argument), for
    callers that cannot allocate device memory; see include/specverify.h."""
    return int(load_library().sv_verify_greedy_noalloc(B, gamma, V, logits, logits_dtype, draft_tokens, out_tokens,
                                                       out_num_accepted, out_status, stream))


def sv_verify_sample_ragged(B, gamma, V, logits, logits_dtype, q, draft_tokens, uniforms, gamma_b, temperature,
                            top_k, top_p, out_tokens, out_num_accepted, out_accept_prob, out_status, workspace,
                            workspace_bytes, stream) -> int:
    return int(load_library().sv_verify_sample_ragged(B, gamma, V, logits, logits_dtype, q, draft_tokens, uniforms,
                                                       gamma_b, float(temperature), int(top_k), float(top_p),
                                                       out_tokens, out_num_accepted, out_accept_prob, out_status,
                                                       workspace, workspace_bytes, stream))


def sv_verify_greedy_ragged(B, gamma, V, logits, logits_dtype, draft_tokens, gamma_b, out_tokens, out_num_accepted,
                            out_status, workspace, workspace_bytes, stream) -> int:
    return int(load_library().sv_verify_greedy_ragged(B, gamma, V, logits, logits_dtype, draft_tokens, gamma_b,
                                                       out_tokens, out_num_accepted, out_status, workspace,
                                                       workspace_bytes, stream))


def sv_truncate_emitted(B, gamma, tokens, num_accepted, stop_tokens, n_stop, max_new, out_num_emitted,
                        stream) -> int:
    return int(load_library().sv_truncate_emitted(B, gamma, tokens, num_accepted, stop_tokens, n_stop, max_new,
                                                   out_num_emitted, stream))


def sv_pointer_device_readable(ptr) -> bool:
    """True if the device reads this address as is (device memory, managed
    memory, or pinned host memory mapped at the same address)."""
    return bool(load_library().sv_pointer_device_readable(ptr))


def sv_last_kernels() -> list:
    """Kernels launched by the last verify call on this thread, in order."""
    names = load_library().sv_last_kernels().decode()
    return names.split(",") if names else []


def sv_set_timing_events(events) -> int:
    """Register three torch.cuda.Event objects (or None to clear) that later
    calls record around their kernels (benchmark hook)."""
    lib = load_library()
    if not events:
        return int(lib.sv_set_timing_events(None, 0))
    arr = (_c_ptr * 3)(*[e.cuda_event for e in events])
    return int(lib.sv_set_timing_events(arr, 3))


# ------------------------------------------------------------ torch wrappers

def _addr(t):
    return None if t is None else t.data_ptr()


def _need_cuda(name, t, dtype=None):
    if t is None:
        return
    if not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor (the library runs on the GPU only)")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    if dtype is not None and t.dtype != dtype:
        raise ValueError(f"{name} must be {dtype}, got {t.dtype}")


def _need_readable(name, t, dtype=None):
    """A CUDA tensor, or a host tensor in pinned memory the device reads at
    the same address (q may stay on the host: the kernels read only the
    entries the method needs)."""
    if t is None or t.is_cuda:
        _need_cuda(name, t, dtype)
        return
    if not t.is_pinned() or not sv_pointer_device_readable(t.data_ptr()):
        raise ValueError(f"{name} must be a CUDA tensor or pinned host memory the device can read")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    if dtype is not None and t.dtype != dtype:
        raise ValueError(f"{name} must be {dtype}, got {t.dtype}")


def alloc_workspace(B: int, gamma: int, V: int, top_k: int = 0, device=None) -> torch.Tensor:
    """A zero-filled device workspace large enough for (B, gamma, V, top_k)."""
    n = sv_workspace_bytes(B, gamma, V, top_k)
    if n == 0 and B > 0:
        raise SvError(SV_ERR_INVALID_ARG, "sv_workspace_bytes")
    return torch.zeros(max(n, 256), dtype=torch.uint8, device=device)


def _stream_handle(device, stream):
    s = stream if stream is not None else torch.cuda.current_stream(device)
    return s.cuda_stream


def verify_sample(logits, q, draft, uniforms, temperature=1.0, top_k=0, top_p=1.0, *, workspace=None,
                  stream=None, want_accept_prob=True, outputs=None, gamma_b=None):
    """Speculative-sampling verify of a batch on the GPU.

    logits [B, gamma+1, V] (float32 / bfloat16 / float16), q [B, gamma, V]
    float32 (or None: deterministic drafts, q one-hot at each drafted token),
    draft [B, gamma] int32, uniforms [B, gamma+1] float32, all CUDA tensors
    except q, which may also be a pinned host tensor (read in place: only
    q(d_i), the kept candidates and a rejected sequence's residual row cross
    the host link).  gamma_b [B] int32 (CUDA) makes the round ragged:
    sequence b drafted only gamma_b[b] tokens (sv_verify_sample_ragged).
    Returns (out_tokens [B, gamma+1] int32, n_accepted [B] int32, accept_prob
    [B, gamma] float32 or None, status [B] int32).
    """
    B, G1, V = logits.shape
    G = G1 - 1
    dev = logits.device
    _need_cuda("logits", logits)
    if logits.dtype not in _TORCH_DTYPE:
        raise ValueError(f"unsupported logits dtype {logits.dtype}")
    _need_readable("q", q if G > 0 else None, torch.float32)
    _need_cuda("draft", draft if G > 0 else None, torch.int32)
    _need_cuda("uniforms", uniforms, torch.float32)
    if outputs is None:
        out_tokens = torch.empty(B, G1, dtype=torch.int32, device=dev)
        out_n = torch.empty(B, dtype=torch.int32, device=dev)
        out_a = torch.empty(B, G, dtype=torch.float32, device=dev) if want_accept_prob and G > 0 else None
        out_status = torch.empty(B, dtype=torch.int32, device=dev)
    else:
        out_tokens, out_n, out_a, out_status = outputs
    if workspace is None:
        workspace = alloc_workspace(B, G, V, top_k, dev)
    if gamma_b is None:
        st = sv_verify_sample(B, G, V, _addr(logits), _TORCH_DTYPE[logits.dtype], _addr(q) if G > 0 else None,
                              _addr(draft) if G > 0 else None, _addr(uniforms), temperature, top_k, top_p,
                              _addr(out_tokens), _addr(out_n), _addr(out_a), _addr(out_status),
                              _addr(workspace), workspace.numel(), _stream_handle(dev, stream))
    else:
        _need_cuda("gamma_b", gamma_b, torch.int32)
        st = sv_verify_sample_ragged(B, G, V, _addr(logits), _TORCH_DTYPE[logits.dtype],
                                     _addr(q) if G > 0 else None, _addr(draft) if G > 0 else None, _addr(uniforms),
                                     _addr(gamma_b), temperature, top_k, top_p, _addr(out_tokens), _addr(out_n),
                                     _addr(out_a), _addr(out_status), _addr(workspace), workspace.numel(),
                                     _stream_handle(dev, stream))
    if st != SV_OK:
        raise SvError(st, "sv_verify_sample")
    return out_tokens, out_n, out_a, out_status


def alloc_qlogits_workspace(B: int, gamma: int, V: int, top_k: int = 0, device=None) -> torch.Tensor:
    """A zero-filled device workspace large enough for verify_sample_qlogits."""
    n = sv_qlogits_workspace_bytes(B, gamma, V, top_k)
    if n == 0 and B > 0:
        raise SvError(SV_ERR_INVALID_ARG, "sv_qlogits_workspace_bytes")
    return torch.zeros(max(n, 256), dtype=torch.uint8, device=device)


def verify_sample_qlogits(logits, q_logits, draft, uniforms, temperature=1.0, top_k=0, top_p=1.0, *,
                          workspace=None, stream=None, want_accept_prob=True, outputs=None):
    """Speculative-sampling verify with the draft's proposal given as its
    logits: q_logits [B, gamma, V] (float32 / bfloat16 / float16, CUDA);
    q_i = softmax(q_logits_i / temperature), truncated by top_k / top_p like
    p_i, is formed on the GPU.  Other
    arguments and the result as verify_sample."""
    B, G1, V = logits.shape
    G = G1 - 1
    dev = logits.device
    _need_cuda("logits", logits)
    if logits.dtype not in _TORCH_DTYPE:
        raise ValueError(f"unsupported logits dtype {logits.dtype}")
    if G > 0:
        _need_cuda("q_logits", q_logits)
        if q_logits.dtype not in _TORCH_DTYPE:
            raise ValueError(f"unsupported q_logits dtype {q_logits.dtype}")
    _need_cuda("draft", draft if G > 0 else None, torch.int32)
    _need_cuda("uniforms", uniforms, torch.float32)
    if outputs is None:
        out_tokens = torch.empty(B, G1, dtype=torch.int32, device=dev)
        out_n = torch.empty(B, dtype=torch.int32, device=dev)
        out_a = torch.empty(B, G, dtype=torch.float32, device=dev) if want_accept_prob and G > 0 else None
        out_status = torch.empty(B, dtype=torch.int32, device=dev)
    else:
        out_tokens, out_n, out_a, out_status = outputs
    if workspace is None:
        workspace = alloc_qlogits_workspace(B, G, V, top_k, dev)
    st = sv_verify_sample_qlogits(B, G, V, _addr(logits), _TORCH_DTYPE[logits.dtype],
                                  _addr(q_logits) if G > 0 else None,
                                  _TORCH_DTYPE[q_logits.dtype] if G > 0 else 0,
                                  _addr(draft) if G > 0 else None, _addr(uniforms), temperature, top_k, top_p,
                                  _addr(out_tokens), _addr(out_n), _addr(out_a), _addr(out_status),
                                  _addr(workspace), workspace.numel(), _stream_handle(dev, stream))
    if st != SV_OK:
        raise SvError(st, "sv_verify_sample_qlogits")
    return out_tokens, out_n, out_a, out_status


def verify_greedy(logits, draft, *, workspace=None, stream=None, outputs=None, gamma_b=None):
    """Greedy verify of a batch on the GPU (gamma_b [B] int32 CUDA: a ragged
    round).  Returns (out_tokens, n_accepted, status)."""
    B, G1, V = logits.shape
    G = G1 - 1
    dev = logits.device
    _need_cuda("logits", logits)
    if logits.dtype not in _TORCH_DTYPE:
        raise ValueError(f"unsupported logits dtype {logits.dtype}")
    _need_cuda("draft", draft if G > 0 else None, torch.int32)
    if outputs is None:
        out_tokens = torch.empty(B, G1, dtype=torch.int32, device=dev)
        out_n = torch.empty(B, dtype=torch.int32, device=dev)
        out_status = torch.empty(B, dtype=torch.int32, device=dev)
    else:
        out_tokens, out_n, out_status = outputs
    if workspace is None:
        workspace = alloc_workspace(B, G, V, 0, dev)
    if gamma_b is None:
        st = sv_verify_greedy(B, G, V, _addr(logits), _TORCH_DTYPE[logits.dtype], _addr(draft) if G > 0 else None,
                              _addr(out_tokens), _addr(out_n), _addr(out_status), _addr(workspace),
                              workspace.numel(), _stream_handle(dev, stream))
    else:
        _need_cuda("gamma_b", gamma_b, torch.int32)
        st = sv_verify_greedy_ragged(B, G, V, _addr(logits), _TORCH_DTYPE[logits.dtype],
                                     _addr(draft) if G > 0 else None, _addr(gamma_b), _addr(out_tokens),
                                     _addr(out_n), _addr(out_status), _addr(workspace), workspace.numel(),
                                     _stream_handle(dev, stream))
    if st != SV_OK:
        raise SvError(st, "sv_verify_greedy")
    return out_tokens, out_n, out_status


def truncate_emitted(tokens, n_accepted, stop_tokens=None, max_new=None, *, stream=None):
    """End the round early at stop tokens / a token budget, in place on
    `tokens` [B, gamma+1] int32 (CUDA).  stop_tokens: int32 CUDA tensor of
    token ids (or None); max_new: [B] int32 CUDA tensor (or None).  Returns
    num_emitted [B] int32."""
    B, G1 = tokens.shape
    dev = tokens.device
    _need_cuda("tokens", tokens, torch.int32)
    _need_cuda("n_accepted", n_accepted, torch.int32)
    _need_cuda("stop_tokens", stop_tokens, torch.int32)
    _need_cuda("max_new", max_new, torch.int32)
    out = torch.empty(B, dtype=torch.int32, device=dev)
    n_stop = 0 if stop_tokens is None else stop_tokens.numel()
    st = sv_truncate_emitted(B, G1 - 1, _addr(tokens), _addr(n_accepted), _addr(stop_tokens), n_stop,
                             _addr(max_new), _addr(out), _stream_handle(dev, stream))
    if st != SV_OK:
        raise SvError(st, "sv_truncate_emitted")
    return out
