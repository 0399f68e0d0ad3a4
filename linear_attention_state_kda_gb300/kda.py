"""Thin Python binding of libkda.so (include/kda.h): one function per C entry point.

Argument marshalling only: tensors are passed as raw device pointers with their sizes, on
the current torch CUDA stream; every step of the computation runs in the library's CUDA
kernels. Outputs that the caller does not supply are allocated with torch (plumbing).
Loading fails loudly if the library was not built: there is no fallback.
"""
import ctypes
import os

import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "_build", "libkda.so")

KDA_OK, KDA_ERR_INVALID_ARG, KDA_ERR_UNSUPPORTED, KDA_ERR_WORKSPACE, KDA_ERR_CUDA = range(5)
KDA_F32, KDA_BF16 = 0, 1
DECODE_BETA_LOGIT = 1
CONV_SILU = 1
MAX_WINDOW = 16
STATUS_BAD_SLOT, STATUS_BAD_OFFSETS, STATUS_TIMEOUT = 1, 4, 8

_lib = None


class KdaError(RuntimeError):
    def __init__(self, status, msg):
        super().__init__(f"[kda status {status}] {msg}")
        self.status = status


def lib():
    """The loaded libkda.so (ctypes). Raises if it has not been built."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(LIB_PATH):
        raise RuntimeError(f"libkda.so not found at {LIB_PATH}: build it with "
                           "`python -c 'import __graft_entry__ as g; g.build()'`")
    L = ctypes.CDLL(LIB_PATH)
    P, I, F, Z, I64 = (ctypes.c_void_p, ctypes.c_int, ctypes.c_float, ctypes.c_size_t,
                       ctypes.c_int64)
    L.kda_last_error.restype = ctypes.c_char_p
    L.kda_last_error.argtypes = []
    L.kda_version.restype = ctypes.c_char_p
    L.kda_version.argtypes = []
    L.kda_launch_count.restype = ctypes.c_uint64
    L.kda_launch_count.argtypes = []
    L.kda_chunk_workspace.restype = Z
    L.kda_chunk_workspace.argtypes = [I, I, I, I, I, I]
    L.kda_chunk_prefill.restype = I
    L.kda_chunk_prefill.argtypes = [I, I, I, P, I, I, I, I, F, P, P, P, P, P, P, P, P, P, Z, P,
                                    P]
    L.kda_segment_package.restype = I
    L.kda_segment_package.argtypes = [I, I, I, P, I, I, I, I, P, P, P, P, P, P, P, Z, P, P]
    L.kda_package_scan_workspace.restype = Z
    L.kda_package_scan_workspace.argtypes = [I, I, I, I, I]
    L.kda_package_scan.restype = I
    L.kda_package_scan.argtypes = [I, I, P, I, I, I, I, P, P, P, P, P, P, Z, P, P]
    L.kda_package_scan_noalloc.restype = I
    L.kda_package_scan_noalloc.argtypes = [I, I, P, I, I, I, I, P, P, P, P, P, P, P]
    L.kda_segment_replay.restype = I
    L.kda_segment_replay.argtypes = [I, I, I, P, I, I, I, I, F, P, P, P, P, P, P, P, P, P, Z, P,
                                     P]
    L.kda_chunk_prepare.restype = I
    L.kda_chunk_prepare.argtypes = [I, I, I, P, I, I, I, I, F, P, P, P, P, P, P, Z, P, P]
    L.kda_segment_package_prepared.restype = I
    L.kda_segment_package_prepared.argtypes = [I, I, I, P, I, I, I, I, P, P, P, Z, P, P]
    L.kda_segment_replay_prepared.restype = I
    L.kda_segment_replay_prepared.argtypes = [I, I, I, P, I, I, I, I, P, P, P, P, Z, P, P]
    L.kda_debug_flag_wait.restype = I
    L.kda_debug_flag_wait.argtypes = [I, I, I, P, I, I, I, I, P, P, P, P, Z, ctypes.c_uint64,
                                      P, P]
    L.kda_decode_step.restype = I
    L.kda_decode_step.argtypes = [I, I, I, I, I, F, P, P, P, P, P, P, P, I64, P, P, P]
    L.kda_decode_window.restype = I
    L.kda_decode_window.argtypes = [I, I, I, I, I, I, F, P, P, P, P, P, ctypes.c_uint, P, P, P,
                                    I64, P, P, P]
    L.kda_slot_zero.restype = I
    L.kda_slot_zero.argtypes = [I, P, P, I64, I64, P, P]
    L.kda_slot_copy.restype = I
    L.kda_slot_copy.argtypes = [I, P, P, I64, P, P, I64, I64, P, P]
    L.kda_short_conv.restype = I
    L.kda_short_conv.argtypes = [I, I, I, P, I, I, P, P, ctypes.c_uint, P, P, P, I64, P, P, P]
    _lib = L
    return L


def version():
    return lib().kda_version().decode()


def launch_count():
    """Kernels launched through the library by this process so far."""
    return int(lib().kda_launch_count())


def last_error():
    return lib().kda_last_error().decode()


def _check(st):
    if st != KDA_OK:
        raise KdaError(st, last_error())


def _ptr(t):
    return None if t is None else t.data_ptr()


def _dt(t):
    if t.dtype == torch.bfloat16:
        return KDA_BF16
    if t.dtype == torch.float32:
        return KDA_F32
    raise TypeError(f"unsupported dtype {t.dtype}")


def _stream(stream):
    if stream is None:
        stream = torch.cuda.current_stream()
    return stream.cuda_stream


def _contig(*ts):
    for t in ts:
        if t is not None and not t.is_contiguous():
            raise ValueError("tensors must be contiguous")


def _int32(*ts):
    for t in ts:
        if t is not None and t.dtype != torch.int32:
            raise TypeError("slot ids must be int32 tensors")


def chunk_workspace(dtype, n_ranges, total_tokens, H, dk, dv):
    """kda_chunk_workspace: scratch bytes of the chunked calls (0 if none is needed)."""
    dt = KDA_BF16 if dtype == torch.bfloat16 else KDA_F32
    return int(lib().kda_chunk_workspace(dt, n_ranges, total_tokens, H, dk, dv))


def _chunk_ws(workspace, dtype, n_ranges, T, H, dk, dv, device):
    need = chunk_workspace(dtype, n_ranges, T, H, dk, dv)
    if workspace is None and need > 0:
        workspace = torch.empty(need, dtype=torch.uint8, device=device)
    if workspace is None:
        return None, 0
    return workspace, workspace.numel() * workspace.element_size()


def chunk_prefill(q, k, v, g, beta, cu_seqlens=None, init_state=None, scale=1.0, o=None,
                  final_state=None, want_final=True, status=None, chunk=64, workspace=None,
                  stream=None):
    """kda_chunk_prefill. Returns (o, final_state). `workspace` (uint8 device tensor of at
    least chunk_workspace(...) bytes) is allocated here when not given."""
    _contig(q, k, v, g, beta, cu_seqlens, init_state, o, final_state)
    T, H, dk = k.shape
    dv = v.shape[2]
    n = 1 if cu_seqlens is None else cu_seqlens.numel() - 1
    if o is None:
        o = torch.empty(T, H, dv, dtype=q.dtype, device=q.device)
    if final_state is None and want_final:
        final_state = torch.empty(n, H, dk, dv, dtype=torch.float32, device=q.device)
    ws, ws_bytes = _chunk_ws(workspace, q.dtype, n, T, H, dk, dv, q.device)
    _check(lib().kda_chunk_prefill(_dt(q), n, T, _ptr(cu_seqlens), H, dk, dv, chunk,
                                   float(scale), _ptr(q), _ptr(k), _ptr(v), _ptr(g),
                                   _ptr(beta), _ptr(init_state), _ptr(o), _ptr(final_state),
                                   _ptr(ws), ws_bytes, _ptr(status), _stream(stream)))
    return o, final_state


def segment_package(k, v, g, beta, seg_offsets, M=None, D=None, status=None, chunk=64,
                    workspace=None, stream=None):
    """kda_segment_package. Returns (M, D)."""
    _contig(k, v, g, beta, seg_offsets, M, D)
    T, H, dk = k.shape
    dv = v.shape[2]
    P = seg_offsets.numel() - 1
    if M is None:
        M = torch.empty(P, H, dk, dk, dtype=torch.float32, device=k.device)
    if D is None:
        D = torch.empty(P, H, dk, dv, dtype=torch.float32, device=k.device)
    ws, ws_bytes = _chunk_ws(workspace, k.dtype, P, T, H, dk, dv, k.device)
    _check(lib().kda_segment_package(_dt(k), P, T, _ptr(seg_offsets), H, dk, dv, chunk,
                                     _ptr(k), _ptr(v), _ptr(g), _ptr(beta), _ptr(M), _ptr(D),
                                     _ptr(ws), ws_bytes, _ptr(status), _stream(stream)))
    return M, D


def package_scan_workspace(n_seqs, max_segs_per_seq, H, dk, dv):
    return int(lib().kda_package_scan_workspace(n_seqs, max_segs_per_seq, H, dk, dv))


def package_scan(M, D, seq_seg_offsets, max_segs_per_seq, init_state=None, seg_init=None,
                 final_state=None, want_final=True, workspace=None, status=None, stream=None):
    """kda_package_scan. Returns (seg_init, final_state)."""
    _contig(M, D, seq_seg_offsets, init_state, seg_init, final_state)
    P, H, dk, dv = D.shape
    n = seq_seg_offsets.numel() - 1
    if seg_init is None:
        seg_init = torch.empty(P, H, dk, dv, dtype=torch.float32, device=D.device)
    if final_state is None and want_final:
        final_state = torch.empty(n, H, dk, dv, dtype=torch.float32, device=D.device)
    ws_bytes = package_scan_workspace(n, max_segs_per_seq, H, dk, dv)
    if workspace is None:
        workspace = torch.empty(ws_bytes, dtype=torch.uint8, device=D.device)
    _check(lib().kda_package_scan(n, P, _ptr(seq_seg_offsets), int(max_segs_per_seq), H, dk,
                                  dv, _ptr(M), _ptr(D), _ptr(init_state), _ptr(seg_init),
                                  _ptr(final_state), _ptr(workspace), workspace.numel(),
                                  _ptr(status), _stream(stream)))
    return seg_init, final_state


def package_scan_noalloc(M, D, seq_seg_offsets, max_segs_per_seq, init_state=None,
                         seg_init=None, final_state=None, want_final=True, status=None,
                         stream=None):
    """kda_package_scan_noalloc: the scan with the library's built-in 64 MiB scratch, for
    callers that cannot allocate device memory (pass seg_init / final_state to allocate
    nothing here either). Returns (seg_init, final_state)."""
    _contig(M, D, seq_seg_offsets, init_state, seg_init, final_state)
    P, H, dk, dv = D.shape
    n = seq_seg_offsets.numel() - 1
    if seg_init is None:
        seg_init = torch.empty(P, H, dk, dv, dtype=torch.float32, device=D.device)
    if final_state is None and want_final:
        final_state = torch.empty(n, H, dk, dv, dtype=torch.float32, device=D.device)
    _check(lib().kda_package_scan_noalloc(n, P, _ptr(seq_seg_offsets), int(max_segs_per_seq),
                                          H, dk, dv, _ptr(M), _ptr(D), _ptr(init_state),
                                          _ptr(seg_init), _ptr(final_state), _ptr(status),
                                          _stream(stream)))
    return seg_init, final_state


def segment_replay(q, k, v, g, beta, seg_offsets, seg_init, scale=1.0, o=None,
                   seg_final=None, want_final=False, status=None, chunk=64, workspace=None,
                   stream=None):
    """kda_segment_replay. Returns (o, seg_final)."""
    _contig(q, k, v, g, beta, seg_offsets, seg_init, o, seg_final)
    T, H, dk = k.shape
    dv = v.shape[2]
    P = seg_offsets.numel() - 1
    if o is None:
        o = torch.empty(T, H, dv, dtype=q.dtype, device=q.device)
    if seg_final is None and want_final:
        seg_final = torch.empty(P, H, dk, dv, dtype=torch.float32, device=q.device)
    ws, ws_bytes = _chunk_ws(workspace, q.dtype, P, T, H, dk, dv, q.device)
    _check(lib().kda_segment_replay(_dt(q), P, T, _ptr(seg_offsets), H, dk, dv, chunk,
                                    float(scale), _ptr(q), _ptr(k), _ptr(v), _ptr(g),
                                    _ptr(beta), _ptr(seg_init), _ptr(o), _ptr(seg_final),
                                    _ptr(ws), ws_bytes, _ptr(status), _stream(stream)))
    return o, seg_final


def chunk_prepare(q, k, v, g, beta, offsets=None, scale=1.0, workspace=None, status=None,
                  chunk=64, stream=None):
    """kda_chunk_prepare: per-chunk records of the ranges in `offsets` (q may be None when
    only packages will be built). Returns the workspace tensor holding them."""
    _contig(q, k, v, g, beta, offsets)
    T, H, dk = k.shape
    dv = v.shape[2]
    n = 1 if offsets is None else offsets.numel() - 1
    ws, ws_bytes = _chunk_ws(workspace, k.dtype, n, T, H, dk, dv, k.device)
    _check(lib().kda_chunk_prepare(_dt(k), n, T, _ptr(offsets), H, dk, dv, chunk, float(scale),
                                   _ptr(q), _ptr(k), _ptr(v), _ptr(g), _ptr(beta), _ptr(ws),
                                   ws_bytes, _ptr(status), _stream(stream)))
    return ws


def segment_package_prepared(workspace, seg_offsets, T, H, dk, dv, M=None, D=None,
                             dtype=torch.bfloat16, status=None, chunk=64, stream=None):
    """kda_segment_package_prepared over records from chunk_prepare. Returns (M, D)."""
    _contig(seg_offsets, M, D)
    P = seg_offsets.numel() - 1
    dev = workspace.device
    if M is None:
        M = torch.empty(P, H, dk, dk, dtype=torch.float32, device=dev)
    if D is None:
        D = torch.empty(P, H, dk, dv, dtype=torch.float32, device=dev)
    dt = KDA_BF16 if dtype == torch.bfloat16 else KDA_F32
    _check(lib().kda_segment_package_prepared(dt, P, T, _ptr(seg_offsets), H, dk, dv, chunk,
                                              _ptr(M), _ptr(D), _ptr(workspace),
                                              workspace.numel(), _ptr(status), _stream(stream)))
    return M, D


def segment_replay_prepared(workspace, seg_offsets, seg_init, T, H, dk, dv, o=None,
                            seg_final=None, want_final=False, dtype=torch.bfloat16, status=None,
                            chunk=64, stream=None):
    """kda_segment_replay_prepared over records prepared with q. Returns (o, seg_final)."""
    _contig(seg_offsets, seg_init, o, seg_final)
    P = seg_offsets.numel() - 1
    dev = workspace.device
    if o is None:
        o = torch.empty(T, H, dv, dtype=dtype, device=dev)
    if seg_final is None and want_final:
        seg_final = torch.empty(P, H, dk, dv, dtype=torch.float32, device=dev)
    dt = KDA_BF16 if dtype == torch.bfloat16 else KDA_F32
    _check(lib().kda_segment_replay_prepared(dt, P, T, _ptr(seg_offsets), H, dk, dv, chunk,
                                             _ptr(seg_init), _ptr(o), _ptr(seg_final),
                                             _ptr(workspace), workspace.numel(), _ptr(status),
                                             _stream(stream)))
    return o, seg_final


RECORD_BYTES = 147968  # one (64-token chunk, head) record of the tensor-core chunk path


def record_flags(workspace, n_ranges, T, H):
    """The ready flags after the records in a chunk workspace (an int32 view)."""
    R = (T // 64 + n_ranges) * H
    return workspace[R * RECORD_BYTES:R * RECORD_BYTES + 4 * R].view(torch.int32)


def debug_flag_wait(workspace, seg_offsets, seg_init, T, H, dk, dv, limit_ns, o=None,
                    seg_final=None, want_final=False, status=None, dtype=torch.bfloat16,
                    chunk=64, stream=None):
    """kda_debug_flag_wait: the prepared replay walk, each record gated by its ready flag
    (bounded by limit_ns). Returns (o, seg_final)."""
    _contig(seg_offsets, seg_init, o, seg_final)
    P = seg_offsets.numel() - 1
    dev = workspace.device
    if o is None:
        o = torch.zeros(T, H, dv, dtype=dtype, device=dev)
    if seg_final is None and want_final:
        seg_final = torch.empty(P, H, dk, dv, dtype=torch.float32, device=dev)
    dt = KDA_BF16 if dtype == torch.bfloat16 else KDA_F32
    _check(lib().kda_debug_flag_wait(dt, P, T, _ptr(seg_offsets), H, dk, dv, chunk,
                                     _ptr(seg_init), _ptr(o), _ptr(seg_final), _ptr(workspace),
                                     workspace.numel(), int(limit_ns), _ptr(status),
                                     _stream(stream)))
    return o, seg_final


def decode_step(q, k, v, g, beta, slot_ids, state_pool, scale=1.0, o=None, status=None,
                stream=None):
    """kda_decode_step (state_pool updated in place). Returns o."""
    _contig(q, k, v, g, beta, slot_ids, state_pool, o)
    B, H, dk = k.shape
    dv = v.shape[2]
    if o is None:
        o = torch.empty(B, H, dv, dtype=q.dtype, device=q.device)
    _check(lib().kda_decode_step(_dt(q), B, H, dk, dv, float(scale), _ptr(q), _ptr(k), _ptr(v),
                                 _ptr(g), _ptr(beta), _ptr(slot_ids), _ptr(state_pool),
                                 int(state_pool.shape[0]), _ptr(o), _ptr(status),
                                 _stream(stream)))
    return o


def decode_window(q, k, v, g, beta, read_slots, write_slots, state_pool, scale=1.0,
                  beta_is_logit=False, o=None, status=None, stream=None):
    """kda_decode_window: rows of `window` tokens (write_slots is [batch, window]; q, k, g are
    [batch*window, H, dk] or [batch, window, H, dk], likewise v and beta). Row b reads slot
    read_slots[b] and stores its state after token j into slot write_slots[b, j]. Returns o,
    shaped like v."""
    _contig(q, k, v, g, beta, read_slots, write_slots, state_pool, o)
    _int32(read_slots, write_slots)
    B = read_slots.numel()
    W = write_slots.numel() // B if B else 0
    if write_slots.numel() != B * W:
        raise ValueError("write_slots must hold batch x window ids")
    H, dk = k.shape[-2], k.shape[-1]
    dv = v.shape[-1]
    if k.numel() != B * W * H * dk:
        raise ValueError("k must hold batch x window tokens")
    if o is None:
        o = torch.empty(v.shape, dtype=q.dtype, device=q.device)
    _check(lib().kda_decode_window(_dt(q), B, W, H, dk, dv, float(scale), _ptr(q), _ptr(k),
                                   _ptr(v), _ptr(g), _ptr(beta),
                                   DECODE_BETA_LOGIT if beta_is_logit else 0, _ptr(read_slots),
                                   _ptr(write_slots), _ptr(state_pool),
                                   int(state_pool.shape[0]), _ptr(o), _ptr(status),
                                   _stream(stream)))
    return o


def slot_zero(state_pool, slot_ids=None, n=None, status=None, stream=None):
    """kda_slot_zero: zero the listed slots of state_pool (all of slots 0..n-1 when slot_ids
    is None)."""
    _contig(state_pool, slot_ids)
    _int32(slot_ids)
    if n is None:
        n = slot_ids.numel() if slot_ids is not None else state_pool.shape[0]
    _check(lib().kda_slot_zero(int(n), _ptr(slot_ids), _ptr(state_pool),
                               int(state_pool.shape[0]), int(state_pool[0].numel()),
                               _ptr(status), _stream(stream)))
    return state_pool


def slot_copy(src, src_ids, dst, dst_ids, n=None, status=None, stream=None):
    """kda_slot_copy: dst[dst_ids[i]] = src[src_ids[i]] (None ids mean 0..n-1)."""
    _contig(src, src_ids, dst, dst_ids)
    _int32(src_ids, dst_ids)
    if src[0].numel() != dst[0].numel():
        raise ValueError("src and dst slots differ in size")
    if n is None:
        n = src_ids.numel() if src_ids is not None else dst_ids.numel()
    _check(lib().kda_slot_copy(int(n), _ptr(src), _ptr(src_ids), int(src.shape[0]), _ptr(dst),
                               _ptr(dst_ids), int(dst.shape[0]), int(src[0].numel()),
                               _ptr(status), _stream(stream)))
    return dst


def short_conv(x, weight, cu_seqlens=None, silu=False, read_slots=None, write_slots=None,
               conv_state=None, out=None, status=None, stream=None):
    """kda_short_conv: causal depthwise convolution of x [T, C] with weight [C, W] over the
    packed sequences of cu_seqlens, each starting from the W - 1 inputs in conv_state
    [n_slots, W-1, C] at its read slot and leaving its last W - 1 inputs at its write slot.
    Returns out [T, C]."""
    _contig(x, weight, cu_seqlens, read_slots, write_slots, conv_state, out)
    _int32(cu_seqlens, read_slots, write_slots)
    T, C = x.shape
    W = weight.shape[1]
    n = 1 if cu_seqlens is None else cu_seqlens.numel() - 1
    if out is None:
        out = torch.empty_like(x)
    n_slots = 0 if conv_state is None else int(conv_state.shape[0])
    _check(lib().kda_short_conv(_dt(x), n, T, _ptr(cu_seqlens), C, W, _ptr(x), _ptr(weight),
                                CONV_SILU if silu else 0, _ptr(read_slots), _ptr(write_slots),
                                _ptr(conv_state), n_slots, _ptr(out), _ptr(status),
                                _stream(stream)))
    return out

