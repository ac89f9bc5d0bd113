// TQ-MSE encoder steps shared by the quantize-append kernel and the fused
// decode step (append + attend).
//
// Method: "RoPE-Aware Bit Allocation for KV-Cache Quantization" — review §1
// Key Terms (TQ-MSE: random rotation, then a per-coordinate scalar codebook;
// the norm is kept as side data).  A warp encodes a token: lane L holds codec
// coordinates 4L..4L+3.  Every float operation is an explicit correctly
// rounded intrinsic (no contraction into FMA is possible), in a fixed order,
// so the codes and norms do not depend on the file that includes this header
// or on its compiler flags.
#pragma once

#include <cuda_fp16.h>

#include "bgtq_internal.h"

namespace bgtq {

// Parameter block of the quantize-append kernels.
struct QParams {
    const __half* k;
    const __half* v;
    int t_new, H;
    const int32_t* pos_start;
    uint8_t* kc;
    float* kn;
    uint8_t* vc;
    float* vn;
    int64_t cap;       // positions per sequence
    CacheMap map;      // record location of (sequence, head, position)
    const HeadTab* heads;
    const float* thr;
    const uint32_t* cells;  // code-search cell tables (bulk kernel)
    int cell_words;
    int bk, bv;
    float v_inv_sqrt;
    int32_t* status;
    __half* k_recent;  // fp16 recent-key ring [B][H][recent][128] (recent > 0)
    int64_t recent;
};

// Appends at least this long (and of the widths below) take the
// two-lanes-per-token bulk kernel; it launches it on `s`.
constexpr int kBulkMinTokens = 64;
cudaError_t launch_quantize_append_bulk(const QParams& p, int bk, int bv, int batch, cudaStream_t s);

namespace {

// Randomized Hadamard on the warp's 128 slots of N tokens at once: stages
// h = 1, 2, 4, ..., 64, pair (j, j+h) inside a piece larger than h becomes
// (a + b, a - b).
template <int N>
__device__ __forceinline__ void warp_butterflies_n(float (&x)[N][4], const int (&plog2)[4], int lane) {
#pragma unroll
    for (int h = 1; h <= 2; h <<= 1) {
#pragma unroll
        for (int n = 0; n < N; ++n) {
            float y[4];
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                const int partner = i ^ h;
                const bool active = (1 << plog2[i]) > h;
                y[i] = !active ? x[n][i] : ((i & h) ? __fsub_rn(x[n][partner], x[n][i]) : __fadd_rn(x[n][i], x[n][partner]));
            }
#pragma unroll
            for (int i = 0; i < 4; ++i) x[n][i] = y[i];
        }
    }
#pragma unroll
    for (int h = 4; h < 128; h <<= 1) {
        const int lm = h >> 2;
        float other[N][4];
#pragma unroll
        for (int n = 0; n < N; ++n)
#pragma unroll
            for (int i = 0; i < 4; ++i) other[n][i] = __shfl_xor_sync(0xffffffffu, x[n][i], lm);
#pragma unroll
        for (int n = 0; n < N; ++n)
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                const int j = 4 * lane + i;
                if ((1 << plog2[i]) > h) x[n][i] = (j & h) ? __fsub_rn(other[n][i], x[n][i]) : __fadd_rn(x[n][i], other[n][i]);
            }
    }
}

__device__ __forceinline__ void warp_butterflies(float (&x)[4], const int (&plog2)[4], int lane) {
    float (&xn)[1][4] = *reinterpret_cast<float (*)[1][4]>(&x);
    warp_butterflies_n<1>(xn, plog2, lane);
}

// Thresholds of width w in the compact shared table: entries
// [2^w - 1, 2^(w+1) - 2), i.e. t_w[k] at index 2^w - 1 + k.
constexpr int kThrCompact = 512;

// Encode N tokens held as x[n][4] per lane (already whitened for keys); the
// N tokens go through every step together so their latencies overlap.
// Gives the codes of the lane's four coordinates and the norms rho.  The code
// of u is the number of width-w thresholds <= u (binary search).
template <int N>
__device__ __forceinline__ void warp_encode_n(float (&x)[N][4], const float (&sgn)[4], const int (&plog2)[4],
                                              const float (&inv_sqrt)[4], const int (&width)[4], int n_coded,
                                              const float* s_thr, int (&code)[N][4], float (&rho)[N]) {
    const int lane = threadIdx.x & 31;
#pragma unroll
    for (int n = 0; n < N; ++n)
#pragma unroll
        for (int i = 0; i < 4; ++i) x[n][i] = __fmul_rn(x[n][i], sgn[i]);
    warp_butterflies_n<N>(x, plog2, lane);
    float part[N];
#pragma unroll
    for (int n = 0; n < N; ++n) {
#pragma unroll
        for (int i = 0; i < 4; ++i) x[n][i] = __fmul_rn(x[n][i], inv_sqrt[i]);
        part[n] = __fadd_rn(__fadd_rn(__fmul_rn(x[n][0], x[n][0]), __fmul_rn(x[n][1], x[n][1])),
                            __fadd_rn(__fmul_rn(x[n][2], x[n][2]), __fmul_rn(x[n][3], x[n][3])));
    }
#pragma unroll
    for (int m = 16; m >= 1; m >>= 1)
#pragma unroll
        for (int n = 0; n < N; ++n) part[n] = __fadd_rn(part[n], __shfl_xor_sync(0xffffffffu, part[n], m));
#pragma unroll
    for (int n = 0; n < N; ++n) rho[n] = __fsqrt_rn(__fdiv_rn(part[n], (float)n_coded));
    float u[N][4];
#pragma unroll
    for (int n = 0; n < N; ++n)
#pragma unroll
        for (int i = 0; i < 4; ++i) u[n][i] = rho[n] > 0.0f ? __fdiv_rn(x[n][i], rho[n]) : 0.0f;
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const float* tb = s_thr + (1 << width[i]) - 1;
        int pos[N];
#pragma unroll
        for (int n = 0; n < N; ++n) pos[n] = 0;
        for (int st = (1 << width[i]) >> 1; st >= 1; st >>= 1) {
#pragma unroll
            for (int n = 0; n < N; ++n)
                if (tb[pos[n] + st - 1] <= u[n][i]) pos[n] += st;
        }
#pragma unroll
        for (int n = 0; n < N; ++n) code[n][i] = pos[n];
    }
}

// Per-lane encoder metadata of one head: keys (codec order, whitening,
// rotation pieces, Block-GTQ widths, K record bit positions) or values
// (identity order, one piece of 128, uniform width).
struct EncLane {
    int pl[4], wd[4], src[4];
    float wh[4], sg[4], is[4];
    int kbit[2];
    int n_coded;
};

__device__ __forceinline__ void enc_lane_load(EncLane& e, const HeadTab* ht, bool is_k, int bv, float v_inv_sqrt,
                                              int lane) {
    e.n_coded = is_k ? ht->n_coded : kD;
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const int j = 4 * lane + i;
        const bool coded = j < e.n_coded;
        e.pl[i] = is_k ? (coded ? ht->plog2[j] : 0) : 7;
        e.wd[i] = is_k ? (coded ? ht->width[j] : 0) : bv;
        e.src[i] = is_k ? ht->perm[j] : j;
        e.wh[i] = is_k ? (coded ? ht->whiten[j] : 0.0f) : 1.0f;
        e.sg[i] = is_k ? ht->sign_k[j] : ht->sign_v[j];
        e.is[i] = is_k ? ht->inv_sqrt[j] : v_inv_sqrt;
    }
#pragma unroll
    for (int pr = 0; pr < 2; ++pr) e.kbit[pr] = is_k ? ht->pair_bit[(2 * lane + pr) & (kNB - 1)] : 0;
}

// Stage the thresholds of every width into the compact shared table.
__device__ __forceinline__ void stage_thresholds(float* s_thr, const float* thr, int i0, int stride) {
    for (int i = i0; i < kThrCompact; i += stride) {
        const int w = 31 - __clz(i + 1);
        const int k = i - ((1 << w) - 1);
        s_thr[i] = (w <= kWMax && k < (1 << w) - 1) ? __ldg(thr + 256 * w + k) : INFINITY;
    }
}

// OR the lane's two K code-pair fields into a zeroed K record in shared memory.
__device__ __forceinline__ void pack_k_fields(uint32_t* rec, const int (&code)[4], const EncLane& e, int lane) {
#pragma unroll
    for (int pr = 0; pr < 2; ++pr) {
        const int j = 4 * lane + 2 * pr;
        if (j + 1 < e.n_coded) {
            const int w = e.wd[2 * pr];
            const uint32_t field = (uint32_t)code[2 * pr] | ((uint32_t)code[2 * pr + 1] << w);
            const int wi = e.kbit[pr] >> 5, sh = e.kbit[pr] & 31;
            atomicOr(&rec[wi], field << sh);
            if (sh + 2 * w > 32) atomicOr(&rec[wi + 1], field >> (32 - sh));
        }
    }
}

// OR the lane's four V codes of token parity `par` into a zeroed V pair
// record (and the bits they occupy into `mask`) in shared memory.
__device__ __forceinline__ void pack_v_fields(uint32_t* rec, uint32_t* mask, const int (&code)[4], int par, int bv,
                                              int lane) {
    const uint32_t m1 = (1u << bv) - 1;
#pragma unroll
    for (int k = 0; k < 4; ++k) {
        const int j = 4 * lane + k;
        const int bit = 2 * bv * j + par * bv;
        const int wi = bit >> 5, sh = bit & 31;
        atomicOr(&rec[wi], (uint32_t)code[k] << sh);
        atomicOr(&mask[wi], m1 << sh);
        if (sh + bv > 32) {
            atomicOr(&rec[wi + 1], (uint32_t)code[k] >> (32 - sh));
            atomicOr(&mask[wi + 1], m1 >> (32 - sh));
        }
    }
}

}  // namespace
}  // namespace bgtq
