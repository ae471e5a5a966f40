"""ctypes binding of libpkv.so: argument marshalling only.

Every function here takes torch tensors, checks that shapes and dtypes agree,
and passes raw pointers, sizes and the current CUDA stream to the C ABI
declared in include/pkv.h.  All arithmetic runs in the library's kernels; there
is no fallback: if the library is missing or a call fails, a RuntimeError is
raised.
"""
from __future__ import annotations

import ctypes
import os

import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "_build", "libpkv.so")

PKV_F32, PKV_F16, PKV_BF16 = 0, 1, 2
DTYPE_CODE = {torch.float32: PKV_F32, torch.float16: PKV_F16, torch.bfloat16: PKV_BF16}
KERNEL_AUTO, KERNEL_CUDA_CORE = 0, 1
PREFILL_TCGEN05, PREFILL_WARP_MMA = 0, 1
WIDE_TCGEN05, WIDE_HEAD_SLICES = 0, 1
STATUS_BITS = {1: "bad block id", 2: "bad context length", 4: "bad slot", 8: "bad copy pair",
               16: "wait timeout"}

# name -> (restype, argtypes)
_P, _I, _I64, _F, _SZ = ctypes.c_void_p, ctypes.c_int, ctypes.c_int64, ctypes.c_float, ctypes.c_size_t
_SIGS = {
    "pkv_last_error_string": (ctypes.c_char_p, []),
    "pkv_version": (_I, []),
    "pkv_device_status": (_I, [_P, ctypes.POINTER(ctypes.c_uint32), _I]),
    "pkv_kv_write": (_I, [_P, _P, _P, _P, _P, _I, _I, _I, _I, _I, _I, _P]),
    "pkv_paged_decode_attention": (_I, [_P, _P, _P, _P, _P, _P, _F, _I, _I, _I, _I, _I, _I, _I,
                                        _I, _I, _I, _P, _SZ, _P]),
    "pkv_decode_workspace_bytes": (_SZ, [_I, _I, _I, _I, _I]),
    "pkv_decode_step": (_I, [_P, _P, _P, _P, _P, _P, _P, _P, _F, _I, _I, _I, _I, _I, _I, _I,
                             _I, _I, _I, _P, _SZ, _P]),
    "pkv_paged_decode_grouped": (_I, [_P, _P, _P, _P, _P, _P, _P, _P, _P, _P, _I, _I, _F, _I, _I,
                                      _I, _I, _I, _I, _I, _I, _I, _I, _P, ctypes.c_size_t, _P]),
    "pkv_group_shared_tokens": (_I, [_P, _P, _P, _I, _I, _I, _I, _P]),
    "pkv_paged_prefill_attention": (_I, [_P, _P, _P, _P, _P, _P, _P, _F, _I, _I, _I, _I, _I,
                                         _I, _I, _I, _I, _I, _P]),
    "pkv_paged_decode_attention_noalloc": (_I, [_P, _P, _P, _P, _P, _P, _F, _I, _I, _I, _I, _I,
                                                _I, _I, _I, _I, _I, _P]),
    "pkv_kv_copy_blocks": (_I, [_P, _P, _P, _I, _I, _I, _I, _I, _I, _P]),
    "pkv_kv_swap_blocks": (_I, [_P, _P, _P, _P, _P, _I, _I, _I, _I, _I, _I, _I, _P]),
    "pkv_seq_swap": (_I, [_P, _P, _I64, _P, _I, ctypes.POINTER(_I)]),
    "pkv_seq_add_cached": (_I, [_P, _I64, _P, _I, ctypes.POINTER(_I)]),
    "pkv_seq_register_blocks": (_I, [_P, _I64, _P, _I, ctypes.POINTER(_I)]),
    "pkv_prefix_cache_stats": (_I, [_P, ctypes.POINTER(_I64), ctypes.POINTER(_I64),
                                    ctypes.POINTER(_I64)]),
    "pkv_set_decode_kernel": (_I, [_I]),
    "pkv_selftest_bounded_wait": (_I, [_I, _P, _P]),
    "pkv_set_prefill_kernel": (_I, [_I]),
    "pkv_set_wide_group_kernel": (_I, [_I]),
    "pkv_alloc_create": (_I, [_I, _I, _P, ctypes.POINTER(_P)]),
    "pkv_alloc_destroy": (_I, [_P]),
    "pkv_seq_add": (_I, [_P, _I64, _I]),
    "pkv_seq_append": (_I, [_P, _I64, ctypes.POINTER(_I64), ctypes.POINTER(_I64),
                            ctypes.POINTER(_I64)]),
    "pkv_step_append": (_I, [_P, _P, _I, _P, _P, ctypes.POINTER(_I)]),
    "pkv_step_append_tables": (_I, [_P, _P, _I, _P, _P, ctypes.POINTER(_I), _P, _I, _P]),
    "pkv_seq_fork": (_I, [_P, _I64, _I64]),
    "pkv_seq_free": (_I, [_P, _I64]),
    "pkv_seq_len": (_I, [_P, _I64, ctypes.POINTER(_I)]),
    "pkv_block_table": (_I, [_P, _I64, _P, _I, ctypes.POINTER(_I)]),
    "pkv_block_tables_dense": (_I, [_P, _P, _I, _I, _P, _P]),
    "pkv_refcount": (_I, [_P, _I, ctypes.POINTER(_I)]),
    "pkv_num_free_blocks": (_I, [_P, ctypes.POINTER(_I)]),
    "pkv_stats": (_I, [_P, ctypes.POINTER(_I64), ctypes.POINTER(_I64), ctypes.POINTER(_I64)]),
}

_lib = None


def lib():
    """The loaded libpkv.so (RuntimeError if it has not been built)."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise RuntimeError(
                "libpkv.so is not built (expected %s); run "
                "`python -c 'import __graft_entry__ as g; g.build()'`" % LIB_PATH)
        handle = ctypes.CDLL(LIB_PATH)
        for name, (res, args) in _SIGS.items():
            f = getattr(handle, name)
            f.restype, f.argtypes = res, args
        _lib = handle
    return _lib


class PkvError(RuntimeError):
    def __init__(self, code, where):
        msg = lib().pkv_last_error_string().decode(errors="replace")
        super().__init__("%s failed (status %d): %s" % (where, code, msg))
        self.code = code


class OutOfBlocks(PkvError):
    pass


def _check(rc, where):
    if rc != 0:
        if rc == -7:
            raise OutOfBlocks(rc, where)
        raise PkvError(rc, where)


def _stream(stream):
    if stream is None:
        stream = torch.cuda.current_stream()
    return ctypes.c_void_p(stream.cuda_stream)


def _dev(t: torch.Tensor, name: str):
    if not t.is_cuda:
        raise ValueError("%s must be a CUDA tensor" % name)
    if not t.is_contiguous():
        raise ValueError("%s must be contiguous" % name)
    return ctypes.c_void_p(t.data_ptr())


# ---------------------------------------------------------------------------
# device calls
# ---------------------------------------------------------------------------

def kv_write(k_cache, v_cache, key, value, slot_mapping, stream=None):
    """Store key/value [T, Hkv, D] into the caches [NB, Hkv, B, D] at
    slot_mapping (int64 [T], -1 = skip)."""
    NB, Hkv, B, D = k_cache.shape
    T = key.shape[0]
    if v_cache.shape != k_cache.shape or key.shape != (T, Hkv, D) or value.shape != key.shape:
        raise ValueError("kv_write: shape mismatch")
    if slot_mapping.dtype != torch.int64 or slot_mapping.numel() != T:
        raise ValueError("kv_write: slot_mapping must be int64 [T]")
    if len({k_cache.dtype, v_cache.dtype, key.dtype, value.dtype}) != 1:
        raise ValueError("kv_write: dtypes differ")
    rc = lib().pkv_kv_write(_dev(k_cache, "k_cache"), _dev(v_cache, "v_cache"), _dev(key, "key"),
                            _dev(value, "value"), _dev(slot_mapping, "slot_mapping"), T, NB, Hkv,
                            D, B, DTYPE_CODE[k_cache.dtype], _stream(stream))
    _check(rc, "pkv_kv_write")


def decode_workspace_bytes(num_seqs, num_heads, head_dim, max_context_len, partition_size):
    return int(lib().pkv_decode_workspace_bytes(num_seqs, num_heads, head_dim, max_context_len,
                                                partition_size))


def paged_decode_attention(out, q, k_cache, v_cache, block_tables, context_lens, scale,
                           block_size, num_kv_heads, partition_size=0, workspace=None,
                           stream=None):
    """out [S, Hq, D] = paged decode attention of q [S, Hq, D] over the caches.
    q and out may be CUDA tensors or pinned host tensors (the kernel reads q
    and writes out over the host link); the other tensors are CUDA tensors."""
    S, Hq, D = q.shape
    NB, Hkv, B, Dk = k_cache.shape
    if (Hkv, B, Dk) != (num_kv_heads, block_size, D) or v_cache.shape != k_cache.shape:
        raise ValueError("paged_decode_attention: cache shape mismatch")
    if out.shape != q.shape:
        raise ValueError("paged_decode_attention: out must be [S, Hq, D]")
    if block_tables.dtype != torch.int32 or context_lens.dtype != torch.int32:
        raise ValueError("block_tables and context_lens must be int32")
    if block_tables.dim() != 2 or block_tables.shape[0] != S or context_lens.shape != (S,):
        raise ValueError("block_tables must be [S, max_blocks], context_lens [S]")
    if q.dtype != k_cache.dtype or v_cache.dtype != k_cache.dtype:
        raise ValueError("q, k_cache, v_cache must share a dtype")
    ws_ptr, ws_bytes = ctypes.c_void_p(0), 0
    if workspace is not None:
        ws_ptr, ws_bytes = _dev(workspace, "workspace"), workspace.numel() * workspace.element_size()
    rc = lib().pkv_paged_decode_attention(
        _reachable(out, "out"), _reachable(q, "q"), _dev(k_cache, "k_cache"),
        _dev(v_cache, "v_cache"),
        _dev(block_tables, "block_tables"), _dev(context_lens, "context_lens"), float(scale),
        int(block_size), int(num_kv_heads), S, Hq, D, block_tables.shape[1], NB,
        DTYPE_CODE[q.dtype], DTYPE_CODE[out.dtype], int(partition_size), ws_ptr, ws_bytes,
        _stream(stream))
    _check(rc, "pkv_paged_decode_attention")


def decode_step(out, q, new_k, new_v, k_cache, v_cache, block_tables, context_lens, scale,
                block_size, num_kv_heads, partition_size=0, workspace=None, stream=None):
    """One decode step: new_k/new_v [S, Hkv, D] are written at position
    context_lens[s]-1 of each sequence, then out [S, Hq, D] = paged decode
    attention of q over the updated caches (q and out may be pinned host
    tensors, as in paged_decode_attention)."""
    S, Hq, D = q.shape
    NB, Hkv, B, Dk = k_cache.shape
    if (Hkv, B, Dk) != (num_kv_heads, block_size, D) or v_cache.shape != k_cache.shape:
        raise ValueError("decode_step: cache shape mismatch")
    if out.shape != q.shape or new_k.shape != (S, Hkv, D) or new_v.shape != new_k.shape:
        raise ValueError("decode_step: out must be [S, Hq, D], new_k/new_v [S, Hkv, D]")
    if block_tables.dtype != torch.int32 or context_lens.dtype != torch.int32:
        raise ValueError("block_tables and context_lens must be int32")
    if block_tables.dim() != 2 or block_tables.shape[0] != S or context_lens.shape != (S,):
        raise ValueError("block_tables must be [S, max_blocks], context_lens [S]")
    if not (q.dtype == k_cache.dtype == v_cache.dtype == new_k.dtype == new_v.dtype):
        raise ValueError("q, new_k, new_v, k_cache, v_cache must share a dtype")
    ws_ptr, ws_bytes = ctypes.c_void_p(0), 0
    if workspace is not None:
        ws_ptr, ws_bytes = _dev(workspace, "workspace"), workspace.numel() * workspace.element_size()
    rc = lib().pkv_decode_step(
        _reachable(out, "out"), _reachable(q, "q"), _dev(new_k, "new_k"), _dev(new_v, "new_v"),
        _dev(k_cache, "k_cache"), _dev(v_cache, "v_cache"), _dev(block_tables, "block_tables"),
        _dev(context_lens, "context_lens"), float(scale), int(block_size), int(num_kv_heads), S,
        Hq, D, block_tables.shape[1], NB, DTYPE_CODE[q.dtype], DTYPE_CODE[out.dtype],
        int(partition_size), ws_ptr, ws_bytes, _stream(stream))
    _check(rc, "pkv_decode_step")


def paged_decode_grouped(out, q, k_cache, v_cache, block_tables, context_lens, group_start,
                         shared_tokens, scale, block_size, num_kv_heads, new_k=None, new_v=None,
                         parts=1, workspace=None, max_members=None, stream=None):
    """Decode attention (a decode step when new_k/new_v [S, Hkv, D] are
    given) for groups of consecutive sequences sharing a prefix of physical
    blocks: group i is sequences group_start[i]..group_start[i+1]-1, whose
    first shared_tokens[i] positions use the same table entries.  Same
    result as decode_step / paged_decode_attention for every sequence; q and
    out may likewise be pinned host tensors.
    parts > 1 cuts each group's stage list over that many CTAs (merged in
    the launch); it needs a workspace of
    decode_workspace_bytes(S, Hq, D, parts, 1) bytes.  max_members bounds the
    members of any group (it picks the kernel width: one n8 column tile when
    max_members * G <= 8); None leaves the bound to the library (the
    sequences the other groups leave)."""
    S, Hq, D = q.shape
    NB, Hkv, B, Dk = k_cache.shape
    if (Hkv, B, Dk) != (num_kv_heads, block_size, D) or v_cache.shape != k_cache.shape:
        raise ValueError("paged_decode_grouped: cache shape mismatch")
    if out.shape != q.shape:
        raise ValueError("paged_decode_grouped: out must be [S, Hq, D]")
    if (new_k is None) != (new_v is None):
        raise ValueError("paged_decode_grouped: pass both new_k and new_v, or neither")
    if new_k is not None and (new_k.shape != (S, Hkv, D) or new_v.shape != new_k.shape or
                              new_k.dtype != q.dtype or new_v.dtype != q.dtype):
        raise ValueError("paged_decode_grouped: new_k/new_v must be [S, Hkv, D] in q's dtype")
    for t, name in ((block_tables, "block_tables"), (context_lens, "context_lens"),
                    (group_start, "group_start"), (shared_tokens, "shared_tokens")):
        if t.dtype != torch.int32:
            raise ValueError("%s must be int32" % name)
    G = group_start.shape[0] - 1
    if group_start.dim() != 1 or G < 1 or shared_tokens.shape != (G,):
        raise ValueError("group_start must be [num_groups + 1], shared_tokens [num_groups]")
    if block_tables.dim() != 2 or block_tables.shape[0] != S or context_lens.shape != (S,):
        raise ValueError("block_tables must be [S, max_blocks], context_lens [S]")
    if not (q.dtype == k_cache.dtype == v_cache.dtype):
        raise ValueError("q, k_cache, v_cache must share a dtype")
    nk = _dev(new_k, "new_k") if new_k is not None else ctypes.c_void_p(0)
    nv = _dev(new_v, "new_v") if new_v is not None else ctypes.c_void_p(0)
    ws_ptr, ws_bytes = ctypes.c_void_p(0), 0
    if workspace is not None:
        ws_ptr, ws_bytes = _dev(workspace, "workspace"), workspace.numel() * workspace.element_size()
    rc = lib().pkv_paged_decode_grouped(
        _reachable(out, "out"), _reachable(q, "q"), nk, nv, _dev(k_cache, "k_cache"),
        _dev(v_cache, "v_cache"),
        _dev(block_tables, "block_tables"), _dev(context_lens, "context_lens"),
        _dev(group_start, "group_start"), _dev(shared_tokens, "shared_tokens"), G,
        int(max_members or 0), float(scale),
        int(block_size), int(num_kv_heads), S, Hq, D, block_tables.shape[1], NB,
        DTYPE_CODE[q.dtype], DTYPE_CODE[out.dtype], int(parts), ws_ptr, ws_bytes,
        _stream(stream))
    _check(rc, "pkv_paged_decode_grouped")


def group_shared_tokens(block_tables, context_lens, group_start, block_size):
    """Host helper: for each group, the leading positions whose table
    entries all members hold in common (whole blocks), at most the shortest
    member's context.  CPU int32 tensors in, CPU int32 [num_groups] out."""
    bt = block_tables.to(torch.int32).contiguous()
    cl = context_lens.to(torch.int32).contiguous()
    gs = group_start.to(torch.int32).contiguous()
    out = torch.zeros(max(gs.shape[0] - 1, 0), dtype=torch.int32)
    prepare_group_shared_tokens(bt, cl, gs, block_size, out)()
    return out


def prepare_group_shared_tokens(block_tables, context_lens, group_start, block_size, out):
    """group_shared_tokens on fixed buffers: checks them once (contiguous host
    int32: tables [S, max_blocks], lengths [S], group starts [G + 1], out [G])
    and returns step(), which writes each group's shared positions into out
    and returns it.  The buffers' contents may change between calls, not
    their storage or shapes; step keeps them alive."""
    bufs = (block_tables, context_lens, group_start, out)
    for t, name in zip(bufs, ("block_tables", "context_lens", "group_start", "out")):
        if t.dtype != torch.int32 or t.is_cuda or not t.is_contiguous():
            raise ValueError("group_shared_tokens: %s must be a contiguous host int32 tensor"
                             % name)
    G = group_start.shape[0] - 1
    if block_tables.dim() != 2 or out.numel() < max(G, 0):
        raise ValueError("group_shared_tokens: bad shapes")
    fn = lib().pkv_group_shared_tokens
    args = (ctypes.c_void_p(block_tables.data_ptr()), ctypes.c_void_p(context_lens.data_ptr()),
            ctypes.c_void_p(group_start.data_ptr()), G, block_tables.shape[0],
            block_tables.shape[1], int(block_size), ctypes.c_void_p(out.data_ptr()))

    def step():
        rc = fn(*args)
        if rc:
            _check(rc, "pkv_group_shared_tokens")
        return out
    step.buffers = bufs
    return step


def paged_prefill_attention(out, q, k_cache, v_cache, block_tables, context_lens, query_start,
                            scale, block_size, num_kv_heads, max_query_len=None, stream=None):
    """Causal multi-token attention over the paged cache: rows
    query_start[s]..query_start[s+1]-1 of q ([rows, Hq, D]) are the last
    tokens of sequence s."""
    R, Hq, D = q.shape
    NB, Hkv, B, Dk = k_cache.shape
    S = context_lens.shape[0]
    if (Hkv, B, Dk) != (num_kv_heads, block_size, D) or v_cache.shape != k_cache.shape:
        raise ValueError("paged_prefill_attention: cache shape mismatch")
    if out.shape != q.shape or query_start.dtype != torch.int32 or \
            query_start.shape != (S + 1,) or block_tables.shape[0] != S:
        raise ValueError("paged_prefill_attention: bad out/query_start/table tensors")
    if max_query_len is None:
        raise ValueError("paged_prefill_attention: pass max_query_len (a host integer)")
    rc = lib().pkv_paged_prefill_attention(
        _dev(out, "out"), _dev(q, "q"), _dev(k_cache, "k_cache"), _dev(v_cache, "v_cache"),
        _dev(block_tables, "block_tables"), _dev(context_lens, "context_lens"),
        _dev(query_start, "query_start"), float(scale), int(block_size), int(num_kv_heads), S,
        Hq, D, block_tables.shape[1], NB, int(max_query_len), DTYPE_CODE[q.dtype],
        DTYPE_CODE[out.dtype], _stream(stream))
    _check(rc, "pkv_paged_prefill_attention")


NOALLOC_SCRATCH_BYTES = 16 << 20


def paged_decode_attention_noalloc(out, q, k_cache, v_cache, block_tables, context_lens, scale,
                                   block_size, num_kv_heads, partition_size, stream=None):
    """Split-context decode whose scratch is the library's fixed device array
    (for callers that cannot allocate device memory); q and out may be pinned
    host tensors.  The C declaration in include/pkv.h gives the limits."""
    S, Hq, D = q.shape
    NB, Hkv, B, Dk = k_cache.shape
    if (Hkv, B, Dk) != (num_kv_heads, block_size, D) or v_cache.shape != k_cache.shape:
        raise ValueError("paged_decode_attention_noalloc: cache shape mismatch")
    if out.shape != q.shape or block_tables.dtype != torch.int32 or \
            context_lens.dtype != torch.int32 or block_tables.shape[0] != S:
        raise ValueError("paged_decode_attention_noalloc: bad out/table/length tensors")
    rc = lib().pkv_paged_decode_attention_noalloc(
        _reachable(out, "out"), _reachable(q, "q"), _dev(k_cache, "k_cache"),
        _dev(v_cache, "v_cache"),
        _dev(block_tables, "block_tables"), _dev(context_lens, "context_lens"), float(scale),
        int(block_size), int(num_kv_heads), S, Hq, D, block_tables.shape[1], NB,
        DTYPE_CODE[q.dtype], DTYPE_CODE[out.dtype], int(partition_size), _stream(stream))
    _check(rc, "pkv_paged_decode_attention_noalloc")


def _reachable(t: torch.Tensor, name: str):
    """Address of a CUDA tensor or of a pinned host tensor (which the GPU
    addresses directly)."""
    if not (t.is_cuda or t.is_pinned()):
        raise ValueError("%s must be a CUDA tensor or pinned host memory" % name)
    if not t.is_contiguous():
        raise ValueError("%s must be contiguous" % name)
    return ctypes.c_void_p(t.data_ptr())


def kv_swap_blocks(dst_k, dst_v, src_k, src_v, pairs, stream=None):
    """Copy whole blocks from pool src to pool dst (pairs int64 [P, 2] of
    (src block, dst block)); each pool may live on the GPU or in pinned host
    memory."""
    NS_, Hkv, B, D = src_k.shape
    ND = dst_k.shape[0]
    if dst_k.shape[1:] != src_k.shape[1:] or dst_v.shape != dst_k.shape or \
            src_v.shape != src_k.shape:
        raise ValueError("kv_swap_blocks: pool shapes differ")
    if len({dst_k.dtype, dst_v.dtype, src_k.dtype, src_v.dtype}) != 1:
        raise ValueError("kv_swap_blocks: dtypes differ")
    if pairs.dtype != torch.int64 or pairs.dim() != 2 or pairs.shape[1] != 2:
        raise ValueError("pairs must be int64 [P, 2]")
    rc = lib().pkv_kv_swap_blocks(
        _reachable(dst_k, "dst_k"), _reachable(dst_v, "dst_v"), _reachable(src_k, "src_k"),
        _reachable(src_v, "src_v"),
        _reachable(pairs, "pairs") if pairs.numel() else ctypes.c_void_p(0), pairs.shape[0],
        NS_, ND, Hkv, D, B, DTYPE_CODE[src_k.dtype], _stream(stream))
    _check(rc, "pkv_kv_swap_blocks")


def kv_copy_blocks(k_cache, v_cache, pairs, stream=None):
    """Copy whole physical blocks: pairs is int64 [P, 2] of (src, dst)."""
    NB, Hkv, B, D = k_cache.shape
    if pairs.dtype != torch.int64 or pairs.dim() != 2 or pairs.shape[1] != 2:
        raise ValueError("pairs must be int64 [P, 2]")
    rc = lib().pkv_kv_copy_blocks(_dev(k_cache, "k_cache"), _dev(v_cache, "v_cache"),
                                  _dev(pairs, "pairs") if pairs.numel() else ctypes.c_void_p(0),
                                  pairs.shape[0], NB, Hkv, D, B, DTYPE_CODE[k_cache.dtype],
                                  _stream(stream))
    _check(rc, "pkv_kv_copy_blocks")


def device_status(reset=True, stream=None):
    """OR of the status bits kernels raised since the last reset (syncs)."""
    bits = ctypes.c_uint32(0)
    rc = lib().pkv_device_status(_stream(stream), ctypes.byref(bits), 1 if reset else 0)
    if rc not in (0, -6):
        _check(rc, "pkv_device_status")
    return int(bits.value)


def selftest_bounded_wait(num_ctas, drained, stream=None):
    """Launch the bounded-wait self-test (see include/pkv.h); `drained` is a
    zeroed int32/uint32 CUDA tensor of one element."""
    _check(lib().pkv_selftest_bounded_wait(int(num_ctas), _dev(drained, "drained"),
                                           _stream(stream)), "pkv_selftest_bounded_wait")


def set_decode_kernel(which):
    _check(lib().pkv_set_decode_kernel(int(which)), "pkv_set_decode_kernel")


def set_wide_group_kernel(which):
    """Kernel for unsplit decode of groups of 32 k query heads: 0 the tcgen05
    kernel (default), 1 head slices on the mma.sync kernel."""
    _check(lib().pkv_set_wide_group_kernel(int(which)), "pkv_set_wide_group_kernel")


def set_prefill_kernel(which):
    _check(lib().pkv_set_prefill_kernel(int(which)), "pkv_set_prefill_kernel")


# ---------------------------------------------------------------------------
# host block allocator
# ---------------------------------------------------------------------------

class BlockAllocator:
    """Host-side block manager (refcounts, copy-on-write, slot mapping)."""

    def __init__(self, num_blocks, block_size, free_order=None):
        self.num_blocks, self.block_size = int(num_blocks), int(block_size)
        self._order = None
        ptr = ctypes.c_void_p(0)
        if free_order is not None:
            self._order = torch.as_tensor(free_order, dtype=torch.int32).contiguous()
            if self._order.numel() != self.num_blocks:
                raise ValueError("free_order must hold num_blocks ids")
            ptr = ctypes.c_void_p(self._order.data_ptr())
        h = ctypes.c_void_p(0)
        _check(lib().pkv_alloc_create(self.num_blocks, self.block_size, ptr, ctypes.byref(h)),
               "pkv_alloc_create")
        self._h = h

    def __del__(self):
        h = getattr(self, "_h", None)
        if h is not None and h.value and _lib is not None:
            _lib.pkv_alloc_destroy(h)
            self._h = None

    def add(self, seq, prompt_len):
        _check(lib().pkv_seq_add(self._h, int(seq), int(prompt_len)), "pkv_seq_add")

    def append(self, seq):
        slot, src, dst = ctypes.c_int64(), ctypes.c_int64(), ctypes.c_int64()
        _check(lib().pkv_seq_append(self._h, int(seq), ctypes.byref(slot), ctypes.byref(src),
                                    ctypes.byref(dst)), "pkv_seq_append")
        return slot.value, (None if src.value < 0 else (src.value, dst.value))

    def step_append(self, seqs):
        """Returns (slots int64 [n], cow_pairs int64 [P, 2]) as host tensors."""
        s = torch.as_tensor(list(seqs), dtype=torch.int64).contiguous()
        n = s.numel()
        slots = torch.empty(n, dtype=torch.int64)
        pairs = torch.empty((max(n, 1), 2), dtype=torch.int64)
        npairs = ctypes.c_int(0)
        _check(lib().pkv_step_append(self._h, ctypes.c_void_p(s.data_ptr()), n,
                                     ctypes.c_void_p(slots.data_ptr()),
                                     ctypes.c_void_p(pairs.data_ptr()), ctypes.byref(npairs)),
               "pkv_step_append")
        return slots, pairs[:npairs.value].clone()

    def step_append_tables(self, seqs, slots, pairs, tables, lens):
        """One decode step that patches the caller's dense tables in place.

        seqs: int64 [n]; slots: int64 [n] (out); pairs: int64 [>= n, 2] (out,
        copy-on-write pairs first); tables: int32 [n, max_blocks] and lens:
        int32 [n], holding the batch's tables and lengths from before the
        step (in any host memory, e.g. a view of a pinned staging buffer).
        Returns the number of copy-on-write pairs written."""
        return self.prepare_step_append_tables(seqs, slots, pairs, tables, lens)()

    def prepare_step_append_tables(self, seqs, slots, pairs, tables, lens):
        """Checks the buffers of step_append_tables once and returns step(),
        which runs pkv_step_append_tables on them and returns the number of
        copy-on-write pairs.  Between calls the buffers' contents may change
        (the batch's sequence ids, tables the caller patched); their storage,
        shapes and dtypes must not.  Made for a serving loop that reuses its
        staging buffers every step: a call is then the C function and one
        ctypes call.  step keeps the allocator and the buffers alive."""
        n = seqs.numel()
        for t, dt, name in ((seqs, torch.int64, "seqs"), (slots, torch.int64, "slots"),
                            (pairs, torch.int64, "pairs"), (tables, torch.int32, "tables"),
                            (lens, torch.int32, "lens")):
            if t.dtype != dt or t.is_cuda or not t.is_contiguous():
                raise ValueError("step_append_tables: %s must be contiguous host %s" % (name, dt))
        if slots.numel() < n or pairs.shape[0] < n or tables.shape[0] != n or \
                lens.numel() != n or tables.dim() != 2:
            raise ValueError("step_append_tables: bad output shapes")
        npairs = ctypes.c_int(0)
        fn = lib().pkv_step_append_tables
        args = (self._h, ctypes.c_void_p(seqs.data_ptr()), n, ctypes.c_void_p(slots.data_ptr()),
                ctypes.c_void_p(pairs.data_ptr()), ctypes.byref(npairs),
                ctypes.c_void_p(tables.data_ptr()), tables.shape[1],
                ctypes.c_void_p(lens.data_ptr()))

        def step():
            rc = fn(*args)
            if rc:
                _check(rc, "pkv_step_append_tables")
            return npairs.value
        step.buffers = (self, seqs, slots, pairs, tables, lens)
        return step

    def fork(self, parent, child):
        _check(lib().pkv_seq_fork(self._h, int(parent), int(child)), "pkv_seq_fork")

    def free(self, seq):
        _check(lib().pkv_seq_free(self._h, int(seq)), "pkv_seq_free")

    free_seq = free

    def add_cached(self, seq, tokens):
        """New sequence for prompt `tokens`, reusing cached full blocks of its
        longest matching prefix; returns the number of reused tokens."""
        t = torch.as_tensor(list(tokens), dtype=torch.int32).contiguous()
        got = ctypes.c_int(0)
        _check(lib().pkv_seq_add_cached(self._h, int(seq), ctypes.c_void_p(t.data_ptr()),
                                        t.numel(), ctypes.byref(got)), "pkv_seq_add_cached")
        return got.value

    def register_blocks(self, seq, tokens):
        """Index the full blocks covering `tokens` (a prefix of the sequence)."""
        t = torch.as_tensor(list(tokens), dtype=torch.int32).contiguous()
        got = ctypes.c_int(0)
        _check(lib().pkv_seq_register_blocks(self._h, int(seq), ctypes.c_void_p(t.data_ptr()),
                                             t.numel(), ctypes.byref(got)),
               "pkv_seq_register_blocks")
        return got.value

    def prefix_cache_stats(self):
        a, b, c = ctypes.c_int64(), ctypes.c_int64(), ctypes.c_int64()
        _check(lib().pkv_prefix_cache_stats(self._h, ctypes.byref(a), ctypes.byref(b),
                                            ctypes.byref(c)), "pkv_prefix_cache_stats")
        return a.value, b.value, c.value

    def swap_to(self, other, seq):
        """Move `seq` into allocator `other`; returns the (this block, other
        block) pairs, int64 [n, 2], for kv_swap_blocks."""
        n = max(1, len(self.table(seq)))
        pairs = torch.empty((n, 2), dtype=torch.int64)
        got = ctypes.c_int(0)
        _check(lib().pkv_seq_swap(self._h, other._h, int(seq), ctypes.c_void_p(pairs.data_ptr()),
                                  n, ctypes.byref(got)), "pkv_seq_swap")
        return pairs[:got.value].clone()

    def length(self, seq):
        n = ctypes.c_int()
        _check(lib().pkv_seq_len(self._h, int(seq), ctypes.byref(n)), "pkv_seq_len")
        return n.value

    def table(self, seq):
        n = ctypes.c_int()
        rc = lib().pkv_block_table(self._h, int(seq), ctypes.c_void_p(0), 0, ctypes.byref(n))
        if rc not in (0, -2):
            _check(rc, "pkv_block_table")
        buf = torch.empty(max(n.value, 1), dtype=torch.int32)
        _check(lib().pkv_block_table(self._h, int(seq), ctypes.c_void_p(buf.data_ptr()), n.value,
                                     ctypes.byref(n)), "pkv_block_table")
        return buf[:n.value].tolist()

    def dense_tables(self, seqs, max_blocks):
        s = torch.as_tensor(list(seqs), dtype=torch.int64).contiguous()
        tables = torch.empty((s.numel(), max_blocks), dtype=torch.int32)
        lens = torch.empty(s.numel(), dtype=torch.int32)
        _check(lib().pkv_block_tables_dense(self._h, ctypes.c_void_p(s.data_ptr()), s.numel(),
                                            int(max_blocks), ctypes.c_void_p(tables.data_ptr()),
                                            ctypes.c_void_p(lens.data_ptr())),
               "pkv_block_tables_dense")
        return tables, lens

    def refcount(self, block):
        c = ctypes.c_int()
        _check(lib().pkv_refcount(self._h, int(block), ctypes.byref(c)), "pkv_refcount")
        return c.value

    def num_free(self):
        c = ctypes.c_int()
        _check(lib().pkv_num_free_blocks(self._h, ctypes.byref(c)), "pkv_num_free_blocks")
        return c.value

    def stats(self):
        a, v, u = ctypes.c_int64(), ctypes.c_int64(), ctypes.c_int64()
        _check(lib().pkv_stats(self._h, ctypes.byref(a), ctypes.byref(v), ctypes.byref(u)),
               "pkv_stats")
        return a.value, v.value, u.value
