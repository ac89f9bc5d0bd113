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
// codes and norms are identical to the warp encoder's.
constexpr int kBulkTok = 128;
// Per-thread column of 129 words in dynamic shared memory (the odd stride
// keeps the threads of a warp on distinct banks): first the fp16 key row,
// then the rotated coordinates that the code loops read back.
constexpr int kColWords = 129;
constexpr int kBulkDynSmem = kBulkTok * kColWords * 4;

// Code of coordinate y at width w: the number of width-w thresholds <= y / rho
// (binary search over the sorted thresholds; the steps wider than the width
// are skipped by a uniform predicate, so the loop has a fixed trip count).
__device__ __forceinline__ uint32_t bulk_code(float y, float rho, int w, const float* s_thr) {
    const float u = rho > 0.0f ? __fdiv_rn(y, rho) : 0.0f;
    const float* tb = s_thr + (1 << w) - 1;
    int c = 0;
#pragma unroll
    for (int k = kWMax - 1; k >= 0; --k)
        if (k < w && tb[c + (1 << k) - 1] <= u) c += 1 << k;
    return (uint32_t)c;
}

template <int W>
__device__ __forceinline__ uint32_t bulk_code_w(float y, float rho, const float* s_thr) {
    const float u = rho > 0.0f ? __fdiv_rn(y, rho) : 0.0f;
    const float* tb = s_thr + (1 << W) - 1;
    int c = 0;
#pragma unroll
    for (int k = W - 1; k >= 0; --k)
        if (tb[c + (1 << k) - 1] <= u) c += 1 << k;
    return (uint32_t)c;
}

// Rotation pieces of one token held by one thread (stage h applies to the
// coordinates [0, end[h]); kFull: one piece of 128), the 1/sqrt(piece)
// scaling and the norm tree; returns rho = sqrt(sum y^2 / n).
// Butterfly stage H over the first e coordinates (e a multiple of 2H);
// pairs outside keep their values (selected, not branched, so z stays in
// registers).
template <int H, bool kFull>
__device__ __forceinline__ void bulk_stage(float (&z)[kD], int e) {
#pragma unroll
    for (int blk = 0; blk < kD; blk += 2 * H) {
        const bool act = kFull || blk < e;
#pragma unroll
        for (int i = 0; i < H; ++i) {
            const float a0 = z[blk + i], a1 = z[blk + i + H];
            const float s0 = __fadd_rn(a0, a1), s1 = __fsub_rn(a0, a1);
            z[blk + i] = act ? s0 : a0;
            z[blk + i + H] = act ? s1 : a1;
        }
    }
}

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
    float part[32];
#pragma unroll
    for (int L = 0; L < 32; ++L) {
#pragma unroll
        for (int i = 0; i < 4; ++i) z[4 * L + i] = __fmul_rn(z[4 * L + i], kFull ? v_inv_sqrt : s_is[4 * L + i]);
        part[L] = __fadd_rn(__fadd_rn(__fmul_rn(z[4 * L], z[4 * L]), __fmul_rn(z[4 * L + 1], z[4 * L + 1])),
                            __fadd_rn(__fmul_rn(z[4 * L + 2], z[4 * L + 2]), __fmul_rn(z[4 * L + 3], z[4 * L + 3])));
    }
#pragma unroll
    for (int m = 16; m >= 1; m >>= 1)
#pragma unroll
        for (int L = 0; L < m; ++L) part[L] = __fadd_rn(part[L], part[L + m]);
    return __fsqrt_rn(__fdiv_rn(part[0], (float)n));
}

template <int BK, int BV>
__global__ void __launch_bounds__(kBulkTok) quantize_append_bulk_kernel(QParams p) {
    __shared__ float s_thr[kThrCompact];
    __shared__ float s_ws[kD];   // whitening x sign (keys; 0 past n_coded)
    __shared__ float s_is[kD];   // 1/sqrt(piece) (keys)
    __shared__ float s_sv[kD];   // value signs
    __shared__ uint8_t s_perm[kD];
    __shared__ uint8_t s_width[kD];
    __shared__ uint16_t s_pbit[kNB];
    __shared__ int s_end[7];
    __shared__ uint32_t s_rec[kBulkTok * (4 * BK + 1)];
    __shared__ uint32_t s_vrec[kBulkTok * (8 * BV + 1)];
    extern __shared__ float s_col[];
    const int tid = threadIdx.x;
    const int h = blockIdx.y, b = blockIdx.z;
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");

    // ---- plan-static set-up (thread tid prepares codec coordinate tid)
    const HeadTab* ht = p.heads + h;
    const int nc = ht->n_coded;
    stage_thresholds(s_thr, p.thr, tid, kBulkTok);
    {
        const int j = tid;
        const bool coded = j < nc;
        s_ws[j] = coded ? __fmul_rn(ht->whiten[j], ht->sign_k[j]) : 0.0f;
        s_is[j] = ht->inv_sqrt[j];
        s_sv[j] = ht->sign_v[j];
        s_perm[j] = ht->perm[j];
        s_width[j] = coded ? ht->width[j] : 0;
        if (j < kNB) s_pbit[j] = ht->pair_bit[j];
        if (j < 7) {
            int e = 0;
            for (int i = 0; i < nc; ++i) e += (1 << ht->plog2[i]) > (1 << j);
            s_end[j] = e;
        }
    }
    __syncthreads();
    // pos_start is read before the wait: no kernel of this library writes it
    const int ps = p.pos_start[b];
    asm volatile("griddepcontrol.wait;" ::: "memory");
    if (ps < 0 || (int64_t)ps + p.t_new > p.cap) {
        if (blockIdx.x == 0 && h == 0 && tid == 0 && p.status) atomicOr(p.status, BGTQ_STATUS_APPEND_CAPACITY);
        return;
    }
    const int64_t end = (int64_t)ps + p.t_new;
    const int64_t pos = (int64_t)(ps & ~1) + (int64_t)blockIdx.x * kBulkTok + tid;
    const bool act = pos >= ps && pos < end;
    const size_t unit = (size_t)b * p.H + h;
    const int64_t sl = act ? p.map.slot(b, h, pos) : 0;  // record location of token `pos`
    if (sl < 0 && p.status) atomicOr(p.status, BGTQ_STATUS_PAGE_RANGE);

    // ---- key of token `pos`
    if (act) {
        const uint4* src = reinterpret_cast<const uint4*>(p.k + (unit * p.t_new + (size_t)(pos - ps)) * kD);
        float* col = s_col + tid * kColWords;
        uint32_t* row = reinterpret_cast<uint32_t*>(col);
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
        for (int j = 0; j < kD; ++j) z[j] = j < nc ? __fmul_rn(__half2float(rowh[s_perm[j]]), s_ws[j]) : 0.0f;
        const float rho = bulk_rotate_norm<false>(z, nc, s_end, s_is, p.v_inv_sqrt);
#pragma unroll
        for (int j = 0; j < kD; ++j) col[j] = z[j];
        uint32_t* rec = s_rec + tid * (4 * BK + 1);
#pragma unroll
        for (int i = 0; i < 4 * BK; ++i) rec[i] = 0;
        // codes and packing as a rolled loop over the codec pairs (small code)
#pragma unroll 2
        for (int m = 0; 2 * m < nc; ++m) {
            const int w = s_width[2 * m];
            const uint32_t field = bulk_code(col[2 * m], rho, w, s_thr) | (bulk_code(col[2 * m + 1], rho, w, s_thr) << w);
            const int bit = s_pbit[m];
            const int wi = bit >> 5, sh = bit & 31;
            rec[wi] |= field << sh;
            if (sh + 2 * w > 32) rec[wi + 1] |= field >> (32 - sh);
        }
        if (sl >= 0) {
            uint4* dst = reinterpret_cast<uint4*>(p.kc + sl * (16 * BK));
#pragma unroll
            for (int i = 0; i < BK; ++i) dst[i] = make_uint4(rec[4 * i], rec[4 * i + 1], rec[4 * i + 2], rec[4 * i + 3]);
            p.kn[sl] = rho;
        }
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
        float* col = s_col + tid * kColWords;
#pragma unroll
        for (int j = 0; j < kD; ++j) col[j] = z[j];
        // fields as for an even token (code at bit 2 BV j), shifted up by BV
        // for an odd one; codes by a rolled loop into a shared-memory record
        uint32_t* vr = s_vrec + tid * (8 * BV + 1);
#pragma unroll
        for (int i = 0; i < kW; ++i) vr[i] = 0;
#pragma unroll 4
        for (int j = 0; j < kD; ++j) {
            const uint32_t c = bulk_code_w<BV>(col[j], rho_v, s_thr);
            const int bit = 2 * BV * j;
            vr[bit >> 5] |= c << (bit & 31);
            if ((bit & 31) + BV > 32) vr[(bit >> 5) + 1] |= c >> (32 - (bit & 31));
        }
#pragma unroll
        for (int i = 0; i < kW; ++i) vw[i] = vr[i];
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
            const int bit = 2 * BV * j + par * BV;
            mask[bit >> 5] |= m1 << (bit & 31);
            if ((bit & 31) + BV > 32) mask[(bit >> 5) + 1] |= m1 >> (32 - (bit & 31));
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
    cfg.gridDim = dim3((unsigned)(((int64_t)p.t_new + 1 + kBulkTok - 1) / kBulkTok), (unsigned)p.H, (unsigned)batch);
    cfg.blockDim = dim3(kBulkTok, 1, 1);
    cfg.dynamicSmemBytes = kBulkDynSmem;
    auto go = [&](auto kernel) -> cudaError_t {
        // the per-thread columns exceed the 48 KB default: raise it (cheap; idempotent)
        cudaError_t e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kBulkDynSmem);
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
