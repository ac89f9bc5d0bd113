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
// then the rotated coordinates that the code loops read back.  The quotients
// u = y / rho use the token's reciprocal of rho (see quot), and the code
// searches run at the width of each rotation piece.
constexpr int kColWords = 129;
constexpr int kBulkDynSmem = kBulkTok * kColWords * 4;

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

// Code of quotient u at width W: the number of width-W thresholds <= u, by
// binary search over the sorted thresholds tb (= s_thr + 2^W - 1).
template <int W>
__device__ __forceinline__ uint32_t code_w(float u, const float* tb) {
    int c = 0;
#pragma unroll
    for (int k = W - 1; k >= 0; --k)
        if (tb[c + (1 << k) - 1] <= u) c += 1 << k;
    return (uint32_t)c;
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

// Codes and packing of the key pairs of one rotation piece (codec coordinates
// [j0, j0 + n), all of width W) into the thread's record: four pairs at a time
// so that their threshold searches overlap.
template <int W>
__device__ __forceinline__ void bulk_key_piece(const float* col, int j0, int n, float rho, float r, const float* s_thr,
                                               const uint16_t* s_pbit, uint32_t* rec) {
    const float* tb = s_thr + (1 << W) - 1;
    const int m1 = (j0 + n) >> 1;
    for (int m0 = j0 >> 1; m0 < m1; m0 += 4) {
        uint32_t f[4];
#pragma unroll
        for (int q = 0; q < 4; ++q) {
            const int m = min(m0 + q, m1 - 1);
            f[q] = code_w<W>(quot(col[2 * m], rho, r), tb) | (code_w<W>(quot(col[2 * m + 1], rho, r), tb) << W);
        }
#pragma unroll
        for (int q = 0; q < 4; ++q) {
            if (m0 + q >= m1) break;
            const int bit = s_pbit[m0 + q];
            const int wi = bit >> 5, sh = bit & 31;
            rec[wi] |= f[q] << sh;
            if (sh + 2 * W > 32) rec[wi + 1] |= f[q] >> (32 - sh);
        }
    }
}

template <int BK, int BV>
__global__ void __launch_bounds__(kBulkTok) quantize_append_bulk_kernel(QParams p) {
    __shared__ float s_thr[kThrCompact];
    __shared__ float2 s_pw[kD];  // keys: (whitening x sign, source dim) per codec coordinate (0 past n_coded)
    __shared__ float s_is[kD];   // 1/sqrt(piece) (keys)
    __shared__ float s_sv[kD];   // value signs
    __shared__ uint8_t s_width[kD];
    __shared__ uint8_t s_plog2[kD];
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
        s_pw[j] = make_float2(coded ? __fmul_rn(ht->whiten[j], ht->sign_k[j]) : 0.0f, __int_as_float((int)ht->perm[j]));
        s_is[j] = ht->inv_sqrt[j];
        s_sv[j] = ht->sign_v[j];
        s_width[j] = coded ? ht->width[j] : 0;
        s_plog2[j] = coded ? ht->plog2[j] : 0;
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
    float* col = s_col + tid * kColWords;

    // ---- key of token `pos`
    if (act) {
        const uint4* src = reinterpret_cast<const uint4*>(p.k + (unit * p.t_new + (size_t)(pos - ps)) * kD);
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
        for (int j = 0; j < kD; ++j) {
            const float2 pw = s_pw[j];
            z[j] = __fmul_rn(__half2float(rowh[__float_as_int(pw.y)]), pw.x);
        }
        const float rho = bulk_rotate_norm<false>(z, nc, s_end, s_is, p.v_inv_sqrt);
        const float r = rho > 0.0f ? __frcp_rn(rho) : 0.0f;
        // the rotated coordinates go back to the column (the row is no longer
        // needed): the code loops below index them at run time
#pragma unroll
        for (int j = 0; j < kD; ++j) col[j] = z[j];
        uint32_t* rec = s_rec + tid * (4 * BK + 1);
#pragma unroll
        for (int i = 0; i < 4 * BK; ++i) rec[i] = 0;
        // rotation pieces in codec order, each of one width (uniform loop)
        for (int j = 0; j < nc;) {
            const int w = s_width[j], n = 1 << s_plog2[j];
            switch (w) {
                case 1: bulk_key_piece<1>(col, j, n, rho, r, s_thr, s_pbit, rec); break;
                case 2: bulk_key_piece<2>(col, j, n, rho, r, s_thr, s_pbit, rec); break;
                case 3: bulk_key_piece<3>(col, j, n, rho, r, s_thr, s_pbit, rec); break;
                case 4: bulk_key_piece<4>(col, j, n, rho, r, s_thr, s_pbit, rec); break;
                case 5: bulk_key_piece<5>(col, j, n, rho, r, s_thr, s_pbit, rec); break;
                case 6: bulk_key_piece<6>(col, j, n, rho, r, s_thr, s_pbit, rec); break;
                case 7: bulk_key_piece<7>(col, j, n, rho, r, s_thr, s_pbit, rec); break;
                default: bulk_key_piece<8>(col, j, n, rho, r, s_thr, s_pbit, rec); break;
            }
            j += n;
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
        const float r = rho_v > 0.0f ? __frcp_rn(rho_v) : 0.0f;
#pragma unroll
        for (int j = 0; j < kD; ++j) col[j] = z[j];
        // fields as for an even token (code of dim j at bit 2 BV j), shifted up
        // by BV for an odd one; 16 dims (BV words of the record) at a time
        const float* tb = s_thr + (1 << BV) - 1;
        uint32_t* vr = s_vrec + tid * (8 * BV + 1);
#pragma unroll 1
        for (int g = 0; g < 8; ++g) {
            uint32_t wds[BV];
#pragma unroll
            for (int i = 0; i < BV; ++i) wds[i] = 0;
#pragma unroll
            for (int i = 0; i < 16; ++i) {
                const uint32_t c = code_w<BV>(quot(col[16 * g + i], rho_v, r), tb);
                const int bit = 2 * BV * i;  // compile-time after unrolling
                wds[bit >> 5] |= c << (bit & 31);
                if ((bit & 31) + BV > 32) wds[(bit >> 5) + 1] |= c >> (32 - (bit & 31));
            }
#pragma unroll
            for (int i = 0; i < BV; ++i) vr[BV * g + i] = wds[i];
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
