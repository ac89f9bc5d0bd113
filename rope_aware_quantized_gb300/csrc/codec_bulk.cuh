// Bulk quantize-append (prefill): the encoder with two threads per token
// (kernel template; one translation unit per key width instantiates it).
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
// Bulk append (prefill): two threads encode one token.
//
// Lanes l and l + 16 of a warp share the warp's token l: the lane of half hf
// holds codec coordinates (keys) or dims (values) 64 hf .. 64 hf + 63 in
// registers from the gather to the codes.  A block covers kBulkTok
// consecutive positions from an even position, so the two tokens of every V
// pair record are neighbouring lanes of one half.  All threads of a block
// share one (sequence, head); blockIdx.z runs over the key blocks of every
// sequence and then the value blocks (the hardware dispatches blocks in about
// that order, so an SM mostly runs one half of the code at a time).  The arithmetic is the
// encoder's, operation for operation: whitening then signs (one product, as
// the sign is +-1), the butterfly stages of each rotation piece (the pieces
// larger than h form the prefix [0, E_h) of the codec order, pieces being laid
// out by decreasing size and aligned to their size; the stage of width 64
// pairs the two halves, exchanged by shuffle), the 1/sqrt(piece) scaling, the
// 32-partial norm tree (its first level adds partial L + 16, from the other
// half, to partial L; both halves then finish the same tree), the quotient and
// the threshold count, each code one lookup in the cell tables (see
// cell_code); so codes and norms are identical to the warp encoder's.
constexpr int kBulkTok = 64;       // positions per block
constexpr int kBulkThreads = 2 * kBulkTok;
constexpr int kBulkMinBlocks = 5;  // resident blocks per SM the register budget is cut for
// Per-token fp16 key row in dynamic shared memory: 64 words + 1 (the odd
// stride spreads the tokens of a warp over the banks); the plan's cell
// tables follow the rows.
constexpr int kRowWords = 65;
constexpr int kBulkRowBytes = kBulkTok * kRowWords * 4;
constexpr int kCellBatch = 5;      // 16-byte cell-table loads a thread has in flight during the set-up
constexpr int kBulkPairBatch = 8;  // key pairs whose codes are computed before their fields are merged
// Per-half tables are two rows, the second offset from the first so that the
// two halves of a warp, reading entry i of their own rows at once, hit
// distinct banks: 16 banks for 4- and 8-byte entries, 8 for 16-byte ones.
constexpr int kPwRow = 72;   // float2: 144 words
constexpr int kFRow = 80;    // float: 80 words
constexpr int kCpRow = 34;   // uint4: 136 words
constexpr int kPkRow = 48;   // uint32: 48 words

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
    uint32_t th, base, le;
    asm("ld.shared.v2.u32 {%0, %1}, [%2];" : "=r"(th), "=r"(base) : "r"(addr));
    asm("set.le.u32.f32 %0, %1, %2;" : "=r"(le) : "f"(__uint_as_float(th)), "f"(u));  // all ones when t_c <= u
    return base - le;
}

// OR into a shared-memory word without reading it back
__device__ __forceinline__ void red_or_shared(uint32_t addr, uint32_t v) {
    asm volatile("red.shared.or.b32 [%0], %1;" ::"r"(addr), "r"(v) : "memory");
}

// Butterfly stage H < 64 over this half's 64 coordinates, active on the
// local coordinates [0, e) (e a multiple of 2H, or <= 0, or >= 64).  Small
// stages keep the inactive pairs by selection; large ones skip inactive
// blocks by a branch (the halves of a warp may differ: the lanes of the
// inactive half are masked).
template <int H, bool kFull>
__device__ __forceinline__ void half_stage(float (&z)[64], int e) {
#pragma unroll
    for (int blk = 0; blk < 64; blk += 2 * H) {
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

// Stage 64: pair (j, j + 64) is (this lane's coordinate j, the same local
// coordinate of the other half): a + b in half 0, a - b in half 1, both as
// fma(+-1, own, other) (a product by +-1 is exact, so the one rounding is
// that of the sum or difference).  Every lane of the warp takes part.
__device__ __forceinline__ void half_stage64(float (&z)[64], int hf) {
    const float sg = hf ? -1.0f : 1.0f;
#pragma unroll
    for (int i = 0; i < 64; ++i) {
        const float o = __shfl_xor_sync(0xffffffffu, z[i], 16);
        z[i] = __fmaf_rn(sg, z[i], o);
    }
}

// The 1/sqrt(piece) scaling and rho = sqrt(sum y^2 / n): partial L (L = 16 hf
// + l here) is the scaled coordinates 4L..4L+3 squared and summed; the tree
// adds partial L + m to partial L for m = 16, 8, 4, 2, 1.  Level 16 adds the
// other half's partial (the sum is the same in both lanes); the rest is
// computed by both lanes alike.  Every lane of the warp takes part.
template <bool kFull>
__device__ __forceinline__ float half_scale_norm(float (&z)[64], int n, const float* is, float v_inv_sqrt) {
    float node[16];
#pragma unroll
    for (int l = 0; l < 16; ++l) {
#pragma unroll
        for (int i = 0; i < 4; ++i) z[4 * l + i] = __fmul_rn(z[4 * l + i], kFull ? v_inv_sqrt : is[4 * l + i]);
        const float leaf = __fadd_rn(__fadd_rn(__fmul_rn(z[4 * l], z[4 * l]), __fmul_rn(z[4 * l + 1], z[4 * l + 1])),
                                     __fadd_rn(__fmul_rn(z[4 * l + 2], z[4 * l + 2]), __fmul_rn(z[4 * l + 3], z[4 * l + 3])));
        node[l] = __fadd_rn(leaf, __shfl_xor_sync(0xffffffffu, leaf, 16));
    }
#pragma unroll
    for (int m = 8; m >= 1; m >>= 1)
#pragma unroll
        for (int l = 0; l < m; ++l) node[l] = __fadd_rn(node[l], node[l + m]);
    return __fsqrt_rn(__fdiv_rn(node[0], (float)n));
}

// One half of the key of token `pos` (record slot sl when active).  row: the
// token's column of the key rows; rec: the token's record being assembled.
// Every lane of the warp takes part (inactive tokens encode zeros and store
// nothing).
template <int BK>
__device__ __forceinline__ void bulk_key_half(const QParams& p, int nc, int hf, const int* s_end, const float2* pw,
                                              const float* is, const uint4* cp, const uint32_t* pk, uint32_t* row,
                                              uint32_t* rec, const uint4 (&w4)[8], bool act, size_t unit, int64_t pos,
                                              int64_t end, int64_t sl) {
    if (act && p.recent > 0 && pos >= end - p.recent) {
        // fp16 recent-key ring: the key as given, slot pos mod W
        uint4* rdst = reinterpret_cast<uint4*>(p.k_recent + (unit * p.recent + pos % p.recent) * kD) + 8 * hf;
#pragma unroll
        for (int i = 0; i < 8; ++i) rdst[i] = w4[i];
    }
#pragma unroll
    for (int i = 0; i < 8; ++i) {
        row[32 * hf + 4 * i] = w4[i].x;
        row[32 * hf + 4 * i + 1] = w4[i].y;
        row[32 * hf + 4 * i + 2] = w4[i].z;
        row[32 * hf + 4 * i + 3] = w4[i].w;
    }
#pragma unroll
    for (int i = 0; i < 2 * BK; ++i) rec[2 * BK * hf + i] = 0;
    __syncwarp();
    const __half* rowh = reinterpret_cast<const __half*>(row);
    float z[64];
#pragma unroll
    for (int i = 0; i < 64; ++i) {
        const float2 w = pw[i];
        z[i] = __fmul_rn(__half2float(rowh[__float_as_int(w.y)]), w.x);
    }
    const int off = 64 * hf;
    half_stage<1, false>(z, s_end[0] - off);
    half_stage<2, false>(z, s_end[1] - off);
    half_stage<4, false>(z, s_end[2] - off);
    half_stage<8, false>(z, s_end[3] - off);
    half_stage<16, false>(z, s_end[4] - off);
    half_stage<32, false>(z, s_end[5] - off);
    if (s_end[6] > 0) half_stage64(z, hf);  // a piece of 128 (uniform)
    const float rho = half_scale_norm<false>(z, nc, is, p.v_inv_sqrt);
    const float r = rho > 0.0f ? __frcp_rn(rho) : 0.0f;
    const uint32_t rec_a = (uint32_t)__cvta_generic_to_shared(rec);
    // this half's key pairs m = 32 hf + q in codec order, a batch at a time:
    // codes first (their lookups overlap), then the fields OR-ed into the record
#pragma unroll
    for (int q0 = 0; q0 < 32; q0 += kBulkPairBatch) {
        if (2 * (32 * hf + q0) >= nc) break;
        uint32_t f[kBulkPairBatch], pq[kBulkPairBatch];
#pragma unroll
        for (int q = 0; q < kBulkPairBatch; ++q) {
            const uint4 c4 = cp[q0 + q];
            pq[q] = pk[q0 + q];
            const float a = __uint_as_float(c4.x), bb = __uint_as_float(c4.y), sc = __uint_as_float(c4.z);
            const uint32_t c0 = cell_code(quot(z[2 * (q0 + q)], rho, r), a, bb, sc, c4.w);
            const uint32_t c1 = cell_code(quot(z[2 * (q0 + q) + 1], rho, r), a, bb, sc, c4.w);
            f[q] = c0 | (c1 << ((pq[q] >> 16) & 15u));
        }
#pragma unroll
        for (int q = 0; q < kBulkPairBatch; ++q) {
            if (2 * (32 * hf + q0 + q) >= nc) break;
            const uint32_t wa = rec_a + (pq[q] & 0xffu), sh = (pq[q] >> 8) & 31u;
            red_or_shared(wa, f[q] << sh);
            if (pq[q] >> 31) red_or_shared(wa + 4u, f[q] >> (32u - sh));
        }
    }
    __syncwarp();
    asm volatile("" ::: "memory");
    if (act && sl >= 0) {
        if (hf == 0) {
            uint4* dst = reinterpret_cast<uint4*>(p.kc + sl * (16 * BK));
#pragma unroll
            for (int i = 0; i < BK; ++i) dst[i] = make_uint4(rec[4 * i], rec[4 * i + 1], rec[4 * i + 2], rec[4 * i + 3]);
        } else {
            p.kn[sl] = rho;
        }
    }
}

// One half of the value of token `pos` (dims 64 hf .. 64 hf + 63, which fill
// words 4 BV hf .. 4 BV hf + 4 BV - 1 of the V pair record).  The thread pair
// (even, odd token: lanes l, l ^ 1) of a half shares those words.  Every lane
// of the warp takes part.
template <int BV>
__device__ __forceinline__ void bulk_value_half(const QParams& p, int hf, int par, const float* sv,
                                                const uint32_t* s_cell, uint32_t cell_base, const uint4 (&w4)[8],
                                                bool act, int ps, int64_t pos, int64_t end, int64_t sl) {
    float z[64];
#pragma unroll
    for (int i = 0; i < 8; ++i) {
#pragma unroll
        for (int k = 0; k < 4; ++k) {
            const uint32_t wk = k == 0 ? w4[i].x : k == 1 ? w4[i].y : k == 2 ? w4[i].z : w4[i].w;
            const float f0 = __half2float(__ushort_as_half((unsigned short)(wk & 0xffffu)));
            const float f1 = __half2float(__ushort_as_half((unsigned short)(wk >> 16)));
            z[8 * i + 2 * k] = __fmul_rn(f0, sv[8 * i + 2 * k]);
            z[8 * i + 2 * k + 1] = __fmul_rn(f1, sv[8 * i + 2 * k + 1]);
        }
    }
    half_stage<1, true>(z, 64);
    half_stage<2, true>(z, 64);
    half_stage<4, true>(z, 64);
    half_stage<8, true>(z, 64);
    half_stage<16, true>(z, 64);
    half_stage<32, true>(z, 64);
    half_stage64(z, hf);
    const float rho_v = half_scale_norm<true>(z, kD, nullptr, p.v_inv_sqrt);
    const float r = rho_v > 0.0f ? __frcp_rn(rho_v) : 0.0f;
    const uint32_t* hd = s_cell + 4 * BV;
    const float a = __uint_as_float(hd[0]), bb = __uint_as_float(hd[1]), sc = __uint_as_float(hd[2]);
    const uint32_t tab = cell_base + 8u * hd[3] - 8u * kCellMagicBits;
    // fields as for an even token (code of local dim i at bit 2 BV i), shifted
    // up by BV for an odd one (never past the half's last word)
    constexpr int kHW = 4 * BV;  // words of this half of a V pair record
    uint32_t vw[kHW];
#pragma unroll
    for (int i = 0; i < kHW; ++i) vw[i] = 0;
#pragma unroll
    for (int i = 0; i < 64; ++i) {
        const uint32_t c = cell_code(quot(z[i], rho_v, r), a, bb, sc, tab);
        const int bit = 2 * BV * i;  // compile-time after unrolling
        vw[bit >> 5] |= c << (bit & 31);
        if ((bit & 31) + BV > 32) vw[(bit >> 5) + 1] |= c >> (32 - (bit & 31));
    }
    if (par) {
#pragma unroll
        for (int i = kHW - 1; i >= 0; --i) vw[i] = (vw[i] << BV) | (i ? vw[i - 1] >> (32 - BV) : 0u);
    }
    if (!act) {
#pragma unroll
        for (int i = 0; i < kHW; ++i) vw[i] = 0;
    }
    const bool partner = (pos ^ 1) >= ps && (pos ^ 1) < end;
    uint32_t full[kHW];
#pragma unroll
    for (int i = 0; i < kHW; ++i) full[i] = vw[i] | __shfl_xor_sync(0xffffffffu, vw[i], 1);
    if (!act || sl < 0) return;
    if (hf == 0) p.vn[sl] = rho_v;
    uint32_t* vdst = reinterpret_cast<uint32_t*>(p.vc + (sl >> 1) * (32 * BV)) + kHW * hf;
    if (partner) {
        // the pair is complete: the even token's lane stores this half's words
        if (!par) {
            uint4* d4 = reinterpret_cast<uint4*>(vdst);
#pragma unroll
            for (int i = 0; i < BV; ++i) d4[i] = make_uint4(full[4 * i], full[4 * i + 1], full[4 * i + 2], full[4 * i + 3]);
        }
    } else {
        // half-appended pair: merge this token's bits without reading the record
        constexpr uint32_t m1 = (1u << BV) - 1u;
        uint32_t mask[kHW];
#pragma unroll
        for (int i = 0; i < kHW; ++i) mask[i] = 0;
#pragma unroll
        for (int i = 0; i < 64; ++i) {
            const int bit = 2 * BV * i;
            mask[bit >> 5] |= m1 << (bit & 31);
            if ((bit & 31) + BV > 32) mask[(bit >> 5) + 1] |= m1 >> (32 - (bit & 31));
        }
        if (par) {
#pragma unroll
            for (int i = kHW - 1; i >= 0; --i) mask[i] = (mask[i] << BV) | (i ? mask[i - 1] >> (32 - BV) : 0u);
        }
#pragma unroll
        for (int i = 0; i < kHW; ++i) {
            atomicAnd(vdst + i, ~mask[i]);
            atomicOr(vdst + i, vw[i]);
        }
    }
}

template <int BK, int BV>
__global__ void __launch_bounds__(kBulkThreads, kBulkMinBlocks) quantize_append_bulk_kernel(QParams p) {
    __shared__ float2 s_pw[2 * kPwRow];  // keys: (whitening x sign, source dim) per codec coordinate (0 past n_coded)
    __shared__ float s_is[2 * kFRow];    // 1/sqrt(piece) (keys)
    __shared__ float s_sv[2 * kFRow];    // value signs
    __shared__ uint4 s_cp[2 * kCpRow];   // key pair m: a, b, s of its width's cell table (float bits), table base
    // key pair m: byte offset of its first record word | bit shift in it << 8 |
    // width << 16 | field continues in the next word << 31
    __shared__ uint32_t s_pk[2 * kPkRow];
    __shared__ int s_end[7];
    __shared__ uint32_t s_rec[kBulkTok * (4 * BK + 1)];
    extern __shared__ __align__(16) uint32_t s_dyn[];
    uint32_t* const s_cell = s_dyn + kBulkTok * kRowWords;  // the plan's cell tables
    const int tid = threadIdx.x;
    const int nbz = (int)gridDim.z >> 1;
    const bool is_v = (int)blockIdx.z >= nbz;
    const int h = blockIdx.y, b = (int)blockIdx.z - (is_v ? nbz : 0);
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
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
    const int warp = tid >> 5, lane = tid & 31, hf = lane >> 4;
    const int tk = 16 * warp + (lane & 15);  // the block's token of this lane
    const int64_t end = (int64_t)ps + p.t_new;
    const int64_t pos = (int64_t)(ps & ~1) + (int64_t)blockIdx.x * kBulkTok + tk;
    const bool act = pos >= ps && pos < end;
    const size_t unit = (size_t)b * p.H + h;
    // this half of the token's fp16 row (zeros for an inactive token): issued
    // first, so that the plan-static set-up below runs while it is in flight
    uint4 w4[8];
    if (act) {
        const __half* x = is_v ? p.v : p.k;
        const uint4* src = reinterpret_cast<const uint4*>(x + (unit * p.t_new + (size_t)(pos - ps)) * kD) + 8 * hf;
#pragma unroll
        for (int i = 0; i < 8; ++i) w4[i] = __ldg(src + i);
    } else {
#pragma unroll
        for (int i = 0; i < 8; ++i) w4[i] = make_uint4(0u, 0u, 0u, 0u);
    }
    const int64_t sl = act ? p.map.slot(b, h, pos) : 0;  // record location of token `pos`

    // ---- plan-static set-up (thread tid prepares codec coordinate tid)
    const HeadTab* ht = p.heads + h;
    const int nc = ht->n_coded;
    {
        // the cell tables, 16 bytes at a time: every thread's first kCellBatch
        // loads are issued before any store (one round trip for tables of up
        // to kCellBatch x 2 KB), then what is left, then the last 0-3 words
        const int n4 = p.cell_words >> 2;
        const uint4* src4 = reinterpret_cast<const uint4*>(p.cells);
        uint4* dst4 = reinterpret_cast<uint4*>(s_cell);
        uint4 t[kCellBatch];
#pragma unroll
        for (int k = 0; k < kCellBatch; ++k)
            if (tid + k * kBulkThreads < n4) t[k] = __ldg(src4 + tid + k * kBulkThreads);
#pragma unroll
        for (int k = 0; k < kCellBatch; ++k)
            if (tid + k * kBulkThreads < n4) dst4[tid + k * kBulkThreads] = t[k];
        for (int i = tid + kCellBatch * kBulkThreads; i < n4; i += kBulkThreads) dst4[i] = __ldg(src4 + i);
        if (tid < p.cell_words - 4 * n4) s_cell[4 * n4 + tid] = __ldg(p.cells + 4 * n4 + tid);
    }
    {
        const int j = tid, jh = (j >> 6) * kPwRow + (j & 63), jf = (j >> 6) * kFRow + (j & 63);
        const bool coded = j < nc;
        s_pw[jh] = make_float2(coded ? __fmul_rn(ht->whiten[j], ht->sign_k[j]) : 0.0f, __int_as_float((int)ht->perm[j]));
        s_is[jf] = ht->inv_sqrt[j];
        s_sv[jf] = ht->sign_v[j];
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
        const int m = tid, mc = (m >> 5) * kCpRow + (m & 31), mk = (m >> 5) * kPkRow + (m & 31);
        const int w = 2 * m < nc ? ht->width[2 * m] : 0;
        const uint32_t* hd = s_cell + 4 * w;
        s_cp[mc] = make_uint4(hd[0], hd[1], hd[2], cell_base + 8u * hd[3] - 8u * kCellMagicBits);
        const uint32_t bit = ht->pair_bit[m];  // the pair's 2w-bit field starts here
        s_pk[mk] = 4u * (bit >> 5) | (bit & 31u) << 8 | (uint32_t)w << 16 | (uint32_t)((bit & 31u) + 2u * w > 32u) << 31;
    }
    __syncthreads();
    if (sl < 0 && p.status && hf == 0) atomicOr(p.status, BGTQ_STATUS_PAGE_RANGE);
    if (!is_v)
        bulk_key_half<BK>(p, nc, hf, s_end, s_pw + hf * kPwRow, s_is + hf * kFRow, s_cp + hf * kCpRow, s_pk + hf * kPkRow,
                          s_dyn + tk * kRowWords, s_rec + tk * (4 * BK + 1), w4, act, unit, pos, end, sl);
    else
        bulk_value_half<BV>(p, hf, tk & 1, s_sv + hf * kFRow, s_cell, cell_base, w4, act, ps, pos, end, sl);
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
    cfg.blockDim = dim3(kBulkThreads, 1, 1);
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
