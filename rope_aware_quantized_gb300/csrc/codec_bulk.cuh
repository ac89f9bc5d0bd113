// Bulk quantize-append (prefill): the token-per-thread encoder (kernel
// template; one translation unit per key width instantiates it).
//
// Method: "RoPE-Aware Bit Allocation for KV-Cache Quantization" — review §1
// Key Terms (TQ-MSE rotates then quantises; the packed cache stores
// compressed K/V) and English abstract (per-block integer widths for keys,
// uniform TQ-MSE for values).  Built with --fmad=false like the warp encoder;
// every float operation is an explicit correctly rounded intrinsic.
#pragma once

#include <cuda_fp16.h>

#include "bgtq_internal.h"
#include "encode.cuh"

namespace bgtq {
namespace {


// ---------------------------------------------------------------------------
// Bulk append (prefill): one thread encodes one token.
//
// A block covers kBulkTok consecutive positions starting at an even position,
// so the two tokens of every V pair record belong to neighbouring threads.
// All threads of a block share one (sequence, head), so every loop and branch
// over codec coordinates is uniform across the block.  The arithmetic is the
// encoder's, operation for operation: whitening then signs (one product, as
// the sign is +-1), the butterfly stages of each rotation piece (the pieces
// larger than h form the prefix [0, E_h) of the codec order, pieces being laid
// out by decreasing size and aligned to their size), the 1/sqrt(piece)
// scaling, the 32-partial norm tree, the quotient and the threshold count; so
// codes and norms are identical to the warp encoder's.  A token's 128
// coordinates stay in registers from the gather to the codes; each code is
// one lookup in the cell tables (see cell_code), so no loop indexes them at
// run time.
constexpr int kBulkTok = 128;
constexpr int kBulkMinBlocks = 3;  // resident blocks per SM the register budget is cut for
// Per-thread fp16 key row in dynamic shared memory: 64 words + 1 (the odd
// stride keeps the threads of a warp on distinct banks); the plan's cell
// tables follow the rows.
constexpr int kRowWords = 65;
constexpr int kBulkRowBytes = kBulkTok * kRowWords * 4;
constexpr int kBulkPairBatch = 8;  // key pairs whose codes are computed before their fields are merged

// The quotient y / rho correctly rounded, as __fdiv_rn gives it, from the
// correctly rounded reciprocal r = 1/rho (r = 0 when rho = 0, which makes the
// quotient 0 as the encoder requires): two Newton-Raphson corrections in
// Markstein's form, q' = q + r (y - q rho), each remainder exact by FMA; with
// r correctly rounded the last correction rounds to the correctly rounded
// quotient (P. Markstein, "Computation of elementary functions on the IBM
// RISC System/6000 processor", IBM J. Res. Develop. 34(1), 1990).  The
// encoder's quotients lie in [-sqrt(128), sqrt(128)] and come from fp16 data,
// far from under- and overflow.
__device__ __forceinline__ float quot(float y, float rho, float r) {
    const float q0 = __fmul_rn(y, r);
    const float e0 = __fmaf_rn(-q0, rho, y);
    const float q1 = __fmaf_rn(e0, r, q0);
    const float e1 = __fmaf_rn(-q1, rho, y);
    return __fmaf_rn(e1, r, q1);
}

// Code of quotient u (the number of thresholds <= u) from a width's cell
// table: cell c = round(s sat(a u + b)), the low bits of
// fma(sat(fma(u, a, b)), s, 1.5 2^23) (a non-decreasing function of u, so
// every threshold of a lower cell is <= u and every one of a higher cell is
// > u); each cell holds at most one threshold t_c (+inf if none) and the
// count base_c of the thresholds below it, and the code is base_c + [t_c <= u].
// tab = shared address of the width's first entry - 8 x the bits of 1.5 2^23
// (mod 2^32), so the entry address is tab + 8 x the bits of the second fma.
// The load is a plain function of its address (the tables do not change
// while the kernel runs); its address depends on data loaded after the
// tables were staged, which orders it after the staging.
__device__ __forceinline__ uint32_t cell_code(float u, float a, float b, float s, uint32_t tab) {
    const float v = __saturatef(__fmaf_rn(u, a, b));
    const uint32_t addr = tab + ((uint32_t)__float_as_int(__fmaf_rn(v, s, 12582912.0f)) << 3);
    uint32_t th, base;
    asm("ld.shared.v2.u32 {%0, %1}, [%2];" : "=r"(th), "=r"(base) : "r"(addr));
    return base + (__uint_as_float(th) <= u ? 1u : 0u);
}

// OR into a shared-memory word without reading it back
__device__ __forceinline__ void red_or_shared(uint32_t addr, uint32_t v) {
    asm volatile("red.shared.or.b32 [%0], %1;" ::"r"(addr), "r"(v) : "memory");
}

// Butterfly stage H over the first e coordinates (e a multiple of 2H).  Small
// stages keep the pairs past e by selection (nearly every block is active);
// large ones skip inactive blocks by a branch that is uniform across the block.
template <int H, bool kFull>
__device__ __forceinline__ void bulk_stage(float (&z)[kD], int e) {
#pragma unroll
    for (int blk = 0; blk < kD; blk += 2 * H) {
        if constexpr (kFull) {
#pragma unroll
            for (int i = 0; i < H; ++i) {
                const float a0 = z[blk + i], a1 = z[blk + i + H];
                z[blk + i] = __fadd_rn(a0, a1);
                z[blk + i + H] = __fsub_rn(a0, a1);
            }
        } else if constexpr (H < 8) {
            const bool act = blk < e;
#pragma unroll
            for (int i = 0; i < H; ++i) {
                const float a0 = z[blk + i], a1 = z[blk + i + H];
                const float s0 = __fadd_rn(a0, a1), s1 = __fsub_rn(a0, a1);
                z[blk + i] = act ? s0 : a0;
                z[blk + i + H] = act ? s1 : a1;
            }
        } else {
            if (blk < e) {
#pragma unroll
                for (int i = 0; i < H; ++i) {
                    const float a0 = z[blk + i], a1 = z[blk + i + H];
                    z[blk + i] = __fadd_rn(a0, a1);
                    z[blk + i + H] = __fsub_rn(a0, a1);
                }
            }
        }
    }
}

// Node (L, m) of the norm tree: partial L after the sums of the levels above
// m (m = 32: the leaf, coordinates 4L..4L+3 scaled, squared and summed, the
// scaled coordinates written back); node (L, m) = node (L, 2m) + node (L + m, 2m).
template <bool kFull, int M>
__device__ __forceinline__ float norm_tree(float (&z)[kD], int L, const float* s_is, float v_inv_sqrt) {
    if constexpr (M == 32) {
#pragma unroll
        for (int i = 0; i < 4; ++i) z[4 * L + i] = __fmul_rn(z[4 * L + i], kFull ? v_inv_sqrt : s_is[4 * L + i]);
        return __fadd_rn(__fadd_rn(__fmul_rn(z[4 * L], z[4 * L]), __fmul_rn(z[4 * L + 1], z[4 * L + 1])),
                         __fadd_rn(__fmul_rn(z[4 * L + 2], z[4 * L + 2]), __fmul_rn(z[4 * L + 3], z[4 * L + 3])));
    } else {
        const float a = norm_tree<kFull, 2 * M>(z, L, s_is, v_inv_sqrt);
        const float b = norm_tree<kFull, 2 * M>(z, L + M, s_is, v_inv_sqrt);
        return __fadd_rn(a, b);
    }
}

// Rotation pieces of one token held by one thread (stage h applies to the
// coordinates [0, end[h]); kFull: one piece of 128), the 1/sqrt(piece)
// scaling and the norm tree; returns rho = sqrt(sum y^2 / n).
template <bool kFull>
__device__ __forceinline__ float bulk_rotate_norm(float (&z)[kD], int n, const int* s_end, const float* s_is,
                                                  float v_inv_sqrt) {
    bulk_stage<1, kFull>(z, kFull ? kD : s_end[0]);
    bulk_stage<2, kFull>(z, kFull ? kD : s_end[1]);
    bulk_stage<4, kFull>(z, kFull ? kD : s_end[2]);
    bulk_stage<8, kFull>(z, kFull ? kD : s_end[3]);
    bulk_stage<16, kFull>(z, kFull ? kD : s_end[4]);
    bulk_stage<32, kFull>(z, kFull ? kD : s_end[5]);
    bulk_stage<64, kFull>(z, kFull ? kD : s_end[6]);
    // partial L = the scaled coordinates 4L..4L+3 squared and summed; the tree
    // adds partial L + m to partial L for m = 16, 8, 4, 2, 1.  Evaluated depth
    // first (each sum as soon as both of its operands exist), which keeps few
    // partials live and leaves every sum and its operands as they are.
    return __fsqrt_rn(__fdiv_rn(norm_tree<kFull, 1>(z, 0, s_is, v_inv_sqrt), (float)n));
}

template <int BK, int BV>
__global__ void __launch_bounds__(kBulkTok, kBulkMinBlocks) quantize_append_bulk_kernel(QParams p) {
    __shared__ float2 s_pw[kD];  // keys: (whitening x sign, source dim) per codec coordinate (0 past n_coded)
    __shared__ float s_is[kD];   // 1/sqrt(piece) (keys)
    __shared__ float s_sv[kD];   // value signs
    __shared__ uint4 s_cp[kNB];  // key pair m: a, b, s of its width's cell table (float bits), table base
    __shared__ uint32_t s_pk[kNB];  // key pair m: bit position in the record | width << 16
    __shared__ int s_end[7];
    __shared__ uint32_t s_rec[kBulkTok * (4 * BK + 1)];
    extern __shared__ __align__(16) uint32_t s_dyn[];
    uint32_t* const s_cell = s_dyn + kBulkTok * kRowWords;  // the plan's cell tables
    const int tid = threadIdx.x;
    // blockIdx.z: the key blocks of every sequence, then the value blocks
    // (blocks are dispatched in that order, so an SM runs one half of the code
    // at a time)
    const int nbz = (int)gridDim.z >> 1;
    const bool is_v = (int)blockIdx.z >= nbz;
    const int h = blockIdx.y, b = (int)blockIdx.z - (is_v ? nbz : 0);
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");

    // ---- plan-static set-up (thread tid prepares codec coordinate tid)
    const HeadTab* ht = p.heads + h;
    const int nc = ht->n_coded;
    for (int i = tid; i < p.cell_words; i += kBulkTok) s_cell[i] = __ldg(p.cells + i);
    {
        const int j = tid;
        const bool coded = j < nc;
        s_pw[j] = make_float2(coded ? __fmul_rn(ht->whiten[j], ht->sign_k[j]) : 0.0f, __int_as_float((int)ht->perm[j]));
        s_is[j] = ht->inv_sqrt[j];
        s_sv[j] = ht->sign_v[j];
        // E_h = coordinates in pieces larger than h (a prefix: pieces are laid
        // out by decreasing size); written by the last such coordinate, or by
        // thread 0 when there is none
        const int sz = coded ? 1 << ht->plog2[j] : 0;
        const int sz1 = j + 1 < nc ? 1 << ht->plog2[j + 1] : 0;
#pragma unroll
        for (int st = 0; st < 7; ++st) {
            if (sz > (1 << st) && sz1 <= (1 << st)) s_end[st] = j + 1;
            if (j == 0 && sz <= (1 << st)) s_end[st] = 0;
        }
    }
    const uint32_t cell_base = (uint32_t)__cvta_generic_to_shared(s_cell + kCellHdr);
    __syncthreads();
    if (!is_v && tid < kNB) {
        const int m = tid;
        const int w = 2 * m < nc ? ht->width[2 * m] : 0;
        const uint32_t* hd = s_cell + 4 * w;
        s_cp[m] = make_uint4(hd[0], hd[1], hd[2], cell_base + 8u * hd[3] - 8u * kCellMagicBits);
        s_pk[m] = (uint32_t)ht->pair_bit[m] | ((uint32_t)w << 16);
    }
    __syncthreads();
    // pos_start is read before the wait: no kernel of this library writes it
    const int ps = p.pos_start[b];
    asm volatile("griddepcontrol.wait;" ::: "memory");
    if (ps < 0 || (int64_t)ps + p.t_new > p.cap) {
        if (blockIdx.x == 0 && h == 0 && tid == 0 && p.status) {
            atomicOr(p.status, BGTQ_STATUS_APPEND_CAPACITY);
            debug_in_range(false, p.status);  // positions past the capacity
        }
        return;
    }
    const int64_t end = (int64_t)ps + p.t_new;
    const int64_t pos = (int64_t)(ps & ~1) + (int64_t)blockIdx.x * kBulkTok + tid;
    const bool act = pos >= ps && pos < end;
    const size_t unit = (size_t)b * p.H + h;
    const int64_t sl = act ? p.map.slot(b, h, pos) : 0;  // record location of token `pos`
    if (sl < 0 && p.status) atomicOr(p.status, BGTQ_STATUS_PAGE_RANGE);

    // ---- key of token `pos`
    if (!is_v) {
        if (!act) return;
        uint32_t* row = s_dyn + tid * kRowWords;
        const uint4* src = reinterpret_cast<const uint4*>(p.k + (unit * p.t_new + (size_t)(pos - ps)) * kD);
#pragma unroll
        for (int i = 0; i < 16; ++i) {
            const uint4 w4 = __ldg(src + i);
            row[4 * i] = w4.x;
            row[4 * i + 1] = w4.y;
            row[4 * i + 2] = w4.z;
            row[4 * i + 3] = w4.w;
        }
        if (p.recent > 0 && pos >= end - p.recent) {
            // fp16 recent-key ring: the key as given, slot pos mod W
            uint4* rdst = reinterpret_cast<uint4*>(p.k_recent + (unit * p.recent + pos % p.recent) * kD);
#pragma unroll
            for (int i = 0; i < 16; ++i) rdst[i] = make_uint4(row[4 * i], row[4 * i + 1], row[4 * i + 2], row[4 * i + 3]);
        }
        const __half* rowh = reinterpret_cast<const __half*>(row);
        float z[kD];
#pragma unroll
        for (int j = 0; j < kD; ++j) {
            const float2 pw = s_pw[j];
            z[j] = __fmul_rn(__half2float(rowh[__float_as_int(pw.y)]), pw.x);
        }
        const float rho = bulk_rotate_norm<false>(z, nc, s_end, s_is, p.v_inv_sqrt);
        const float r = rho > 0.0f ? __frcp_rn(rho) : 0.0f;
        uint32_t* rec = s_rec + tid * (4 * BK + 1);
#pragma unroll
        for (int i = 0; i < 4 * BK; ++i) rec[i] = 0;
        const uint32_t rec_a = (uint32_t)__cvta_generic_to_shared(rec);
        // key pairs in codec order, a batch at a time: codes first (their
        // lookups overlap), then the fields OR-ed into the record
#pragma unroll
        for (int m0 = 0; m0 < kNB; m0 += kBulkPairBatch) {
            if (2 * m0 >= nc) break;
            uint32_t f[kBulkPairBatch], pk[kBulkPairBatch];
#pragma unroll
            for (int q = 0; q < kBulkPairBatch; ++q) {
                const int m = m0 + q;
                const uint4 cp = s_cp[m];
                pk[q] = s_pk[m];
                const float a = __uint_as_float(cp.x), bb = __uint_as_float(cp.y), sc = __uint_as_float(cp.z);
                const uint32_t c0 = cell_code(quot(z[2 * m], rho, r), a, bb, sc, cp.w);
                const uint32_t c1 = cell_code(quot(z[2 * m + 1], rho, r), a, bb, sc, cp.w);
                f[q] = c0 | (c1 << (pk[q] >> 16));
            }
#pragma unroll
            for (int q = 0; q < kBulkPairBatch; ++q) {
                if (2 * (m0 + q) >= nc) break;
                const uint32_t w = pk[q] >> 16, bit = pk[q] & 0xffffu;
                const uint32_t wa = rec_a + 4u * (bit >> 5), sh = bit & 31u;
                red_or_shared(wa, f[q] << sh);
                if (sh + 2u * w > 32u) red_or_shared(wa + 4u, f[q] >> (32u - sh));
            }
        }
        asm volatile("" ::: "memory");
        if (sl >= 0) {
            uint4* dst = reinterpret_cast<uint4*>(p.kc + sl * (16 * BK));
#pragma unroll
            for (int i = 0; i < BK; ++i) dst[i] = make_uint4(rec[4 * i], rec[4 * i + 1], rec[4 * i + 2], rec[4 * i + 3]);
            p.kn[sl] = rho;
        }
        return;
    }

    // ---- value of token `pos`: the thread pair (even, odd) shares a record
    constexpr int kW = 8 * BV;  // words of a V pair record
    uint32_t vw[kW];
#pragma unroll
    for (int i = 0; i < kW; ++i) vw[i] = 0;
    float rho_v = 0.0f;
    const int par = tid & 1;
    if (act) {
        const uint4* src = reinterpret_cast<const uint4*>(p.v + (unit * p.t_new + (size_t)(pos - ps)) * kD);
        float z[kD];
#pragma unroll
        for (int i = 0; i < 16; ++i) {
            const uint4 w4 = __ldg(src + i);
#pragma unroll
            for (int k = 0; k < 4; ++k) {
                const uint32_t wk = k == 0 ? w4.x : k == 1 ? w4.y : k == 2 ? w4.z : w4.w;
                const float f0 = __half2float(__ushort_as_half((unsigned short)(wk & 0xffffu)));
                const float f1 = __half2float(__ushort_as_half((unsigned short)(wk >> 16)));
                z[8 * i + 2 * k] = __fmul_rn(f0, s_sv[8 * i + 2 * k]);
                z[8 * i + 2 * k + 1] = __fmul_rn(f1, s_sv[8 * i + 2 * k + 1]);
            }
        }
        rho_v = bulk_rotate_norm<true>(z, kD, s_end, s_is, p.v_inv_sqrt);
        const float r = rho_v > 0.0f ? __frcp_rn(rho_v) : 0.0f;
        const uint32_t* hd = s_cell + 4 * BV;
        const float a = __uint_as_float(hd[0]), bb = __uint_as_float(hd[1]), sc = __uint_as_float(hd[2]);
        const uint32_t tab = cell_base + 8u * hd[3] - 8u * kCellMagicBits;
        // fields as for an even token (code of dim j at bit 2 BV j), shifted up
        // by BV for an odd one
#pragma unroll
        for (int j = 0; j < kD; ++j) {
            const uint32_t c = cell_code(quot(z[j], rho_v, r), a, bb, sc, tab);
            const int bit = 2 * BV * j;  // compile-time after unrolling
            vw[bit >> 5] |= c << (bit & 31);
            if ((bit & 31) + BV > 32) vw[(bit >> 5) + 1] |= c >> (32 - (bit & 31));
        }
        if (par) {
#pragma unroll
            for (int i = kW - 1; i >= 0; --i) vw[i] = (vw[i] << BV) | (i ? vw[i - 1] >> (32 - BV) : 0u);
        }
        if (sl >= 0) p.vn[sl] = rho_v;
    }
    const bool partner = (pos ^ 1) >= ps && (pos ^ 1) < end;
    uint32_t full[kW];
#pragma unroll
    for (int i = 0; i < kW; ++i) full[i] = vw[i] | __shfl_xor_sync(0xffffffffu, vw[i], 1);
    if (!act || sl < 0) return;
    uint32_t* vdst = reinterpret_cast<uint32_t*>(p.vc + (sl >> 1) * (32 * BV));
    if (partner) {
        // the pair is complete: the even thread stores the first half, the odd the second
        uint4* d4 = reinterpret_cast<uint4*>(vdst + par * (kW / 2));
#pragma unroll
        for (int i = 0; i < kW / 8; ++i) {
            const int o = 4 * i, q = kW / 2 + 4 * i;  // compile-time indices; the half is selected
            d4[i] = make_uint4(par ? full[q] : full[o], par ? full[q + 1] : full[o + 1], par ? full[q + 2] : full[o + 2],
                               par ? full[q + 3] : full[o + 3]);
        }
    } else {
        // half-appended pair: merge this token's bits without reading the record
        constexpr uint32_t m1 = (1u << BV) - 1u;
        uint32_t mask[kW];
#pragma unroll
        for (int i = 0; i < kW; ++i) mask[i] = 0;
#pragma unroll
        for (int j = 0; j < kD; ++j) {
            const int bit = 2 * BV * j;  // the even token's fields; shifted up by BV for an odd one
            mask[bit >> 5] |= m1 << (bit & 31);
            if ((bit & 31) + BV > 32) mask[(bit >> 5) + 1] |= m1 >> (32 - (bit & 31));
        }
        if (par) {
#pragma unroll
            for (int i = kW - 1; i >= 0; --i) mask[i] = (mask[i] << BV) | (i ? mask[i - 1] >> (32 - BV) : 0u);
        }
#pragma unroll
        for (int i = 0; i < kW; ++i) {
            atomicAnd(vdst + i, ~mask[i]);
            atomicOr(vdst + i, vw[i]);
        }
    }
}

}  // namespace

// Launch the bulk kernel for key width BK (instantiated in codec_bulk_k<BK>.cu).
template <int BK>
cudaError_t launch_bulk_bk(const QParams& p, int bv, int batch, cudaStream_t s);

template <int BK>
cudaError_t launch_bulk_bk_impl(const QParams& p, int bv, int batch, cudaStream_t s) {
    cudaLaunchConfig_t cfg = {};
    cfg.stream = s;
    cudaLaunchAttribute attr;
    attr.id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr.val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = &attr;
    cfg.numAttrs = 1;
    // blocks start at even positions: one more token covers an odd start
    // z: key blocks of every sequence, then value blocks
    if (2 * (int64_t)batch > 65535) return cudaErrorInvalidValue;
    cfg.gridDim = dim3((unsigned)(((int64_t)p.t_new + 1 + kBulkTok - 1) / kBulkTok), (unsigned)p.H, (unsigned)(2 * batch));
    cfg.blockDim = dim3(kBulkTok, 1, 1);
    const int dyn = kBulkRowBytes + 4 * p.cell_words;
    cfg.dynamicSmemBytes = (size_t)dyn;
    auto go = [&](auto kernel) -> cudaError_t {
        // the key rows and cell tables may exceed the 48 KB default: raise it (cheap; idempotent)
        cudaError_t e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, dyn);
        return e != cudaSuccess ? e : cudaLaunchKernelEx(&cfg, kernel, p);
    };
    switch (bv) {
        case 1: return go(quantize_append_bulk_kernel<BK, 1>);
        case 2: return go(quantize_append_bulk_kernel<BK, 2>);
        case 3: return go(quantize_append_bulk_kernel<BK, 3>);
        case 4: return go(quantize_append_bulk_kernel<BK, 4>);
        default: return cudaErrorInvalidValue;
    }
}

}  // namespace bgtq
