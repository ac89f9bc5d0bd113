"""Block-GTQ packed-cache decode path for GB300 (sm_103a).

Python binding of the C ABI in ``include/bgtq.h``.  Every function here only
marshals arguments (numpy arrays for host buffers, torch CUDA tensors for
device buffers) and calls the library of the same name; all of the path's
arithmetic runs in ``libbgtq.so``.  The library must be built
(``rope_aware_quantized_gb300.build.build()``); there is no fallback.

Method: "RoPE-Aware Bit Allocation for KV-Cache Quantization" (English
abstract; paper review §1 Key Terms, §3 Method & Key Results).
"""

from __future__ import annotations

import ctypes as C

import numpy as np

from ._native import BgtqCache, BgtqHeadTables, lib

HEAD_DIM = 128
BGTQ_PLAN_HOST_ONLY = 1
STATUS_APPEND_CAPACITY = 1
STATUS_SEQLEN_CAPACITY = 2
STATUS_PAGE_RANGE = 4


class BgtqError(RuntimeError):
    def __init__(self, code: int, message: str):
        super().__init__(f"bgtq error {code}: {message}")
        self.code = code


def _check(rc: int):
    if rc != 0:
        raise BgtqError(rc, lib().bgtq_last_error().decode())


def _ptr(x) -> int | None:
    if x is None:
        return None
    if isinstance(x, np.ndarray):
        return x.ctypes.data
    return x.data_ptr()


def _stream(stream) -> int | None:
    if stream is None:
        import torch
        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, int):
        return stream
    return stream.cuda_stream


# ----------------------------------------------------------------------------- allocation

def bgtq_alloc_bits(calib_fp16: np.ndarray, bits_per_key: int, b_max: int = 8, rope_layout: int = 0):
    """Block-GTQ widths of one (layer, KV head) -> (bits uint8[64], energy float64[64])."""
    x = np.ascontiguousarray(np.asarray(calib_fp16, dtype=np.float16))
    if x.ndim != 2 or x.shape[1] != HEAD_DIM:
        raise ValueError("calibration keys must be [n][128] float16")
    bits = np.zeros(HEAD_DIM // 2, dtype=np.uint8)
    energy = np.zeros(HEAD_DIM // 2, dtype=np.float64)
    _check(lib().bgtq_alloc_bits(x.ctypes.data, x.shape[0], HEAD_DIM, bits_per_key, b_max, rope_layout,
                                 bits.ctypes.data, energy.ctypes.data))
    return bits, energy


# ----------------------------------------------------------------------------- plan

class Plan:
    """Owner of a bgtq_plan* (codec tables of one layer)."""

    def __init__(self, handle: int, n_kv_heads: int, group: int, bits_per_key: int, v_bits: int):
        self.handle = handle
        self.n_kv_heads = n_kv_heads
        self.group = group
        self.bits_per_key = bits_per_key
        self.v_bits = v_bits

    def destroy(self):
        if self.handle:
            _check(lib().bgtq_plan_destroy(self.handle))
            self.handle = None

    def __del__(self):
        try:
            self.destroy()
        except Exception:
            pass

    def head_tables(self, head: int) -> dict:
        t = BgtqHeadTables()
        _check(lib().bgtq_plan_get_head(self.handle, head, C.byref(t)))

        def arr(p, n, dt):
            return np.ctypeslib.as_array(p, shape=(n,)).astype(dt)
        return {
            "n_coded": t.n_coded,
            "perm": arr(t.perm, 128, np.int64),
            "width": arr(t.width, 128, np.int64),
            "piece": arr(t.piece, 128, np.int64),
            "sign_k": arr(t.sign_k, 128, np.float32),
            "sign_v": arr(t.sign_v, 128, np.float32),
            "whiten": arr(t.whiten, 128, np.float32),
            "dewhiten": arr(t.dewhiten, 128, np.float32),
            "slot_pair": arr(t.slot_pair, 64, np.int64).reshape(4, 16),
            "slot_offset": arr(t.slot_offset, 64, np.int64).reshape(4, 16),
        }

    def codebook(self, width: int):
        cp = C.POINTER(C.c_float)()
        tp = C.POINTER(C.c_float)()
        n = C.c_int()
        _check(lib().bgtq_plan_get_codebook(self.handle, width, C.byref(cp), C.byref(tp), C.byref(n)))
        cent = np.ctypeslib.as_array(cp, shape=(n.value,)).copy()
        thr = np.ctypeslib.as_array(tp, shape=(max(n.value - 1, 0),)).copy() if n.value > 1 else np.zeros(0, np.float32)
        return cent, thr

    def code(self, width: int, u) -> np.ndarray:
        """Codes of the quotients u at one width through the plan's code-search
        cell tables (host): the number of thresholds <= u."""
        uu = np.ascontiguousarray(np.asarray(u, dtype=np.float32).reshape(-1))
        out = np.empty(uu.shape, dtype=np.int32)
        _check(lib().bgtq_plan_code(self.handle, width, uu.ctypes.data, uu.size, out.ctypes.data))
        return out


def bgtq_plan_create(block_bits, energy, group: int, bits_per_key: int, v_bits: int, seed: int,
                     rope_layout: int = 0, host_only: bool = False) -> Plan:
    """Codec tables of one layer from per-head widths [H][64] and energies [H][64]."""
    bb = np.ascontiguousarray(np.asarray(block_bits, dtype=np.uint8).reshape(-1, 64))
    en = np.ascontiguousarray(np.asarray(energy, dtype=np.float64).reshape(-1, 64))
    h = C.c_void_p()
    _check(lib().bgtq_plan_create(C.byref(h), HEAD_DIM, bb.shape[0], group, bits_per_key, v_bits,
                                  bb.ctypes.data, en.ctypes.data, C.c_uint64(seed & ((1 << 64) - 1)),
                                  rope_layout, BGTQ_PLAN_HOST_ONLY if host_only else 0))
    return Plan(h.value, bb.shape[0], group, bits_per_key, v_bits)


def bgtq_plan_save(plan: Plan) -> bytes:
    """The plan as a versioned, checksummed byte record (its defining inputs)."""
    n = C.c_size_t()
    _check(lib().bgtq_plan_save(plan.handle, None, 0, C.byref(n)))
    buf = C.create_string_buffer(n.value)
    _check(lib().bgtq_plan_save(plan.handle, buf, n.value, C.byref(n)))
    return buf.raw[:n.value]


def bgtq_plan_load(data: bytes, host_only: bool = False) -> Plan:
    """A plan rebuilt from a bgtq_plan_save record."""
    data = bytes(data)
    h = C.c_void_p()
    _check(lib().bgtq_plan_load(C.byref(h), data, len(data), BGTQ_PLAN_HOST_ONLY if host_only else 0))
    # the record's header holds the shape: read it back the same way the library does
    H, G, bpk, bv = (int.from_bytes(data[12 + 4 * i:16 + 4 * i], "little") for i in range(4))
    return Plan(h.value, H, G, bpk, bv)


def bgtq_cache_bytes(plan: Plan, batch: int, capacity: int):
    kb, vb, nb = C.c_size_t(), C.c_size_t(), C.c_size_t()
    _check(lib().bgtq_cache_bytes(plan.handle, batch, capacity, C.byref(kb), C.byref(vb), C.byref(nb)))
    return kb.value, vb.value, nb.value


class Cache:
    """One layer's packed cache in caller-owned torch CUDA tensors.

    Contiguous (page_tokens = 0): [batch][H][capacity] records.  Paged
    (page_tokens = P > 0): pools of n_pages pages of P tokens and a page table
    [batch][capacity / P] (int32, device); by default n_pages = batch *
    capacity / P and sequence b's page i is page b * (capacity / P) + i;
    write `page_table` in place (its rows: pool page of each P positions,
    -1 = unmapped) to map them otherwise."""

    def __init__(self, plan: Plan, batch: int, capacity: int, device="cuda", recent: int = 0,
                 page_tokens: int = 0, n_pages: int = 0):
        """recent = W > 0 adds an fp16 recent-key buffer of W keys per (sequence, KV head)."""
        import torch
        if capacity % 2:
            raise ValueError("capacity must be even")
        self.batch, self.capacity, self.recent, self.page_tokens = batch, capacity, recent, page_tokens
        self.page_table = None
        if page_tokens:
            if capacity % page_tokens:
                raise ValueError("a paged cache needs capacity to be a multiple of page_tokens")
            self.max_pages = capacity // page_tokens
            self.n_pages = n_pages or batch * self.max_pages
            kb, vb, nb = bgtq_cache_bytes(plan, self.n_pages, page_tokens)
            ident = torch.arange(batch * self.max_pages, dtype=torch.int32, device=device)
            self.page_table = torch.where(ident < self.n_pages, ident, torch.full_like(ident, -1))
            self.page_table = self.page_table.view(batch, self.max_pages).contiguous()
        else:
            self.max_pages, self.n_pages = 0, 0
            kb, vb, nb = bgtq_cache_bytes(plan, batch, capacity)
        self.k_codes = torch.zeros(kb, dtype=torch.uint8, device=device)
        self.v_codes = torch.zeros(vb, dtype=torch.uint8, device=device)
        self.k_norm = torch.zeros(nb // 4, dtype=torch.float32, device=device)
        self.v_norm = torch.zeros(nb // 4, dtype=torch.float32, device=device)
        rb = batch * plan.n_kv_heads * recent * HEAD_DIM * 2
        self.k_recent = torch.zeros(max(rb // 2, 8), dtype=torch.float16, device=device)
        self.desc = self._desc(0, 0, 0, 0, 0)
        self._per_seq = (kb // max(batch, 1), vb // max(batch, 1), nb // max(batch, 1), rb // max(batch, 1))

    def _desc(self, ko, vo, no, ro, po) -> BgtqCache:
        pt = self.page_table
        return BgtqCache(self.k_codes.data_ptr() + ko, self.k_norm.data_ptr() + no, self.v_codes.data_ptr() + vo,
                         self.v_norm.data_ptr() + no, self.capacity,
                         self.k_recent.data_ptr() + ro if self.recent else None, self.recent,
                         pt.data_ptr() + po if pt is not None else None, self.max_pages, self.page_tokens,
                         self.n_pages)

    def sequence_view(self, b: int) -> "CacheView":
        """Descriptor of sequence b alone (batch 1), per the documented layout."""
        kb, vb, nb, rb = self._per_seq
        if self.page_table is not None:  # same pools, row b of the page table
            return CacheView(self._desc(0, 0, 0, b * rb, b * self.max_pages * 4), self.capacity)
        return CacheView(self._desc(b * kb, b * vb, b * nb, b * rb, 0), self.capacity)

    def nbytes(self) -> int:
        return sum(t.numel() * t.element_size() for t in (self.k_codes, self.v_codes, self.k_norm, self.v_norm)) + \
            (self.k_recent.numel() * 2 if self.recent else 0)


class CacheView:
    """A batch-1 descriptor into a Cache (no memory of its own)."""

    def __init__(self, desc: BgtqCache, capacity: int):
        self.desc = desc
        self.batch = 1
        self.capacity = capacity


# ----------------------------------------------------------------------------- device entry points

def bgtq_quantize_append(plan: Plan, k_fp16, v_fp16, pos_start, cache: Cache, status=None, stream=None):
    """k/v: [B][H][T_new][128] float16 CUDA tensors; pos_start: [B] int32 CUDA tensor."""
    b, h, t_new, d = k_fp16.shape
    if d != HEAD_DIM or tuple(v_fp16.shape) != tuple(k_fp16.shape):
        raise ValueError("k and v must be [B][H][T_new][128]")
    if not (k_fp16.is_contiguous() and v_fp16.is_contiguous()):
        raise ValueError("k and v must be contiguous")
    _check(lib().bgtq_quantize_append(plan.handle, _stream(stream), _ptr(k_fp16), _ptr(v_fp16), b, t_new,
                                      _ptr(pos_start), C.byref(cache.desc), _ptr(status)))


def bgtq_decode_attn_workspace(plan: Plan, batch: int, max_len: int) -> int:
    n = C.c_size_t()
    _check(lib().bgtq_decode_attn_workspace(plan.handle, batch, max_len, C.byref(n)))
    return n.value


def bgtq_decode_attn(plan: Plan, q_fp16, cache: Cache, seq_lens, max_len: int, out, workspace,
                     softmax_scale: float | None = None, status=None, stream=None):
    """q: [B][H*G][128] float16; out: same shape, float16 or float32; workspace: uint8 CUDA tensor."""
    import torch
    batch = q_fp16.shape[0]
    if out.dtype == torch.float32:
        out_dtype = 1
    elif out.dtype == torch.float16:
        out_dtype = 0
    else:
        raise ValueError("out must be float16 or float32")
    scale = (1.0 / HEAD_DIM ** 0.5) if softmax_scale is None else softmax_scale
    _check(lib().bgtq_decode_attn(plan.handle, _stream(stream), _ptr(q_fp16), C.byref(cache.desc), _ptr(seq_lens),
                                  max_len, batch, _ptr(out), out_dtype, scale, _ptr(workspace),
                                  workspace.numel() * workspace.element_size(), _ptr(status)))


def bgtq_decode_step(plan: Plan, q_fp16, k_new, v_new, pos_new, cache: Cache, seq_lens, max_len: int, out,
                     workspace, softmax_scale: float | None = None, status=None, stream=None):
    """One decode step of a layer in one launch: append the new token
    (k_new/v_new: [B][H][128] float16 at pos_new: [B] int32), then attend
    (q: [B][H*G][128] float16 over seq_lens tokens); out as bgtq_decode_attn."""
    import torch
    batch = q_fp16.shape[0]
    if out.dtype == torch.float32:
        out_dtype = 1
    elif out.dtype == torch.float16:
        out_dtype = 0
    else:
        raise ValueError("out must be float16 or float32")
    if k_new.shape[-1] != HEAD_DIM or tuple(v_new.shape) != tuple(k_new.shape) or k_new.numel() != batch * plan.n_kv_heads * HEAD_DIM:
        raise ValueError("k_new and v_new must be [B][H][128]")
    if not (k_new.is_contiguous() and v_new.is_contiguous()):
        raise ValueError("k_new and v_new must be contiguous")
    scale = (1.0 / HEAD_DIM ** 0.5) if softmax_scale is None else softmax_scale
    _check(lib().bgtq_decode_step(plan.handle, _stream(stream), _ptr(q_fp16), _ptr(k_new), _ptr(v_new), _ptr(pos_new),
                                  C.byref(cache.desc), _ptr(seq_lens), max_len, batch, _ptr(out), out_dtype, scale,
                                  _ptr(workspace), workspace.numel() * workspace.element_size(), _ptr(status)))


def bgtq_decode_attn_noalloc(plan: Plan, q_fp16, cache: Cache, seq_lens, max_len: int, out,
                             softmax_scale: float | None = None, status=None, stream=None):
    """bgtq_decode_attn without a workspace, for callers that cannot allocate
    device memory; its merge scratch is the library's built-in 2 MiB array
    (calls that overlap on the GPU race)."""
    import torch
    batch = q_fp16.shape[0]
    if out.dtype == torch.float32:
        out_dtype = 1
    elif out.dtype == torch.float16:
        out_dtype = 0
    else:
        raise ValueError("out must be float16 or float32")
    scale = (1.0 / HEAD_DIM ** 0.5) if softmax_scale is None else softmax_scale
    _check(lib().bgtq_decode_attn_noalloc(plan.handle, _stream(stream), _ptr(q_fp16), C.byref(cache.desc),
                                          _ptr(seq_lens), max_len, batch, _ptr(out), out_dtype, scale, _ptr(status)))


def bgtq_logit_mae(plan: Plan, q_fp16, k_fp16, cache, t: int, out, softmax_scale: float | None = None, stream=None):
    """RoPE-logit fidelity: out [B][H*G] float32 = mean over positions 0..t-1 of
    |scale q.k - scale q.khat| (k_fp16: [B][H][t][128], the appended keys)."""
    batch = q_fp16.shape[0]
    if not k_fp16.is_contiguous() or k_fp16.shape[-1] != HEAD_DIM or k_fp16.shape[-2] != t:
        raise ValueError("k must be a contiguous [B][H][t][128] tensor")
    scale = (1.0 / HEAD_DIM ** 0.5) if softmax_scale is None else softmax_scale
    _check(lib().bgtq_logit_mae(plan.handle, _stream(stream), _ptr(q_fp16), _ptr(k_fp16), C.byref(cache.desc), t,
                                batch, scale, _ptr(out)))


def bgtq_prefill_attn(plan: Plan, q_fp16, k_fp16, v_fp16, cache: Cache, out, softmax_scale: float | None = None,
                      status=None, stream=None):
    """Prefill of a prompt into an empty cache: causal attention over the prompt's own K/V into
    `out` and the packed records of positions 0 .. T-1 into `cache`.
    q: [B][H*G][T][128] float16; k, v: [B][H][T][128] float16; out: like q, float16 or float32."""
    import torch
    b, hq, t, d = q_fp16.shape
    if d != HEAD_DIM or tuple(k_fp16.shape) != (b, plan.n_kv_heads, t, d) or tuple(v_fp16.shape) != tuple(k_fp16.shape):
        raise ValueError("q must be [B][H*G][T][128], k and v [B][H][T][128]")
    if tuple(out.shape) != tuple(q_fp16.shape):
        raise ValueError("out must have the shape of q")
    if not all(x.is_contiguous() for x in (q_fp16, k_fp16, v_fp16, out)):
        raise ValueError("q, k, v and out must be contiguous")
    if out.dtype == torch.float32:
        out_dtype = 1
    elif out.dtype == torch.float16:
        out_dtype = 0
    else:
        raise ValueError("out must be float16 or float32")
    scale = (1.0 / HEAD_DIM ** 0.5) if softmax_scale is None else softmax_scale
    _check(lib().bgtq_prefill_attn(plan.handle, _stream(stream), _ptr(q_fp16), _ptr(k_fp16), _ptr(v_fp16), b, t,
                                   C.byref(cache.desc), _ptr(out), out_dtype, scale, _ptr(status)))


def bgtq_prefill_chunk_workspace(plan: Plan, batch: int, max_prefix: int) -> int:
    n = C.c_size_t()
    _check(lib().bgtq_prefill_chunk_workspace(plan.handle, batch, max_prefix, C.byref(n)))
    return n.value


def bgtq_prefill_chunk_attn(plan: Plan, q_fp16, k_fp16, v_fp16, pos_start, cache: Cache, out,
                            max_prefix: int | None = None, workspace=None, softmax_scale: float | None = None,
                            status=None, stream=None):
    """A later chunk of a prompt onto a cache holding pos_start[b] tokens of sequence b: the
    chunk's packed records into `cache` (an append at pos_start) and attention of every chunk
    row over the cached prefix (as stored) and the chunk's own K/V so far into `out`.
    q: [B][H*G][C][128] float16; k, v: [B][H][C][128] float16; pos_start: [B] int32 CUDA
    tensor; out: like q, float16 or float32.  max_prefix bounds pos_start (read from it when
    None); workspace: a uint8 CUDA tensor of bgtq_prefill_chunk_workspace bytes (allocated
    here when None)."""
    import torch
    b, hq, t, d = q_fp16.shape
    if d != HEAD_DIM or tuple(k_fp16.shape) != (b, plan.n_kv_heads, t, d) or tuple(v_fp16.shape) != tuple(k_fp16.shape):
        raise ValueError("q must be [B][H*G][C][128], k and v [B][H][C][128]")
    if tuple(out.shape) != tuple(q_fp16.shape):
        raise ValueError("out must have the shape of q")
    if tuple(pos_start.shape) != (b,) or pos_start.dtype != torch.int32:
        raise ValueError("pos_start must be an int32 tensor of shape [B]")
    if not all(x.is_contiguous() for x in (q_fp16, k_fp16, v_fp16, out)):
        raise ValueError("q, k, v and out must be contiguous")
    if out.dtype == torch.float32:
        out_dtype = 1
    elif out.dtype == torch.float16:
        out_dtype = 0
    else:
        raise ValueError("out must be float16 or float32")
    if max_prefix is None:
        max_prefix = max(0, int(pos_start.max().item())) if b else 0
    if workspace is None:
        workspace = torch.empty(max(bgtq_prefill_chunk_workspace(plan, b, max_prefix), 1), dtype=torch.uint8,
                                device=q_fp16.device)
    scale = (1.0 / HEAD_DIM ** 0.5) if softmax_scale is None else softmax_scale
    _check(lib().bgtq_prefill_chunk_attn(plan.handle, _stream(stream), _ptr(q_fp16), _ptr(k_fp16), _ptr(v_fp16), b,
                                         t, _ptr(pos_start), max_prefix, C.byref(cache.desc), _ptr(out), out_dtype,
                                         scale, _ptr(workspace), workspace.numel(), _ptr(status)))


def bgtq_dequant_debug(plan: Plan, cache: Cache, b: int, head: int, t0: int, t1: int, k_out=None, v_out=None,
                       codec_domain: bool = False, stream=None):
    _check(lib().bgtq_dequant_debug(plan.handle, _stream(stream), C.byref(cache.desc), cache.batch, b, head, t0, t1,
                                    _ptr(k_out), _ptr(v_out), 1 if codec_domain else 0))


__all__ = [
    "BgtqError", "Plan", "Cache", "CacheView", "bgtq_alloc_bits", "bgtq_plan_create", "bgtq_cache_bytes",
    "bgtq_quantize_append", "bgtq_decode_attn_workspace", "bgtq_decode_attn", "bgtq_decode_step",
    "bgtq_decode_attn_noalloc", "bgtq_logit_mae", "bgtq_prefill_attn", "bgtq_prefill_chunk_workspace", "bgtq_prefill_chunk_attn",
    "bgtq_plan_save", "bgtq_plan_load", "bgtq_dequant_debug",
]
