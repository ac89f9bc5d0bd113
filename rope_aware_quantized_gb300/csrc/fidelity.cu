// RoPE-logit fidelity diagnostic: the mean absolute error of the attention
// logits computed from the packed keys against the keys as given.
//
// Method: "RoPE-Aware Bit Allocation for KV-Cache Quantization" — review §3
// Method & Key Results (Block-GTQ lowers the error of the RoPE logits against
// uniform TQ-MSE at matched bit budgets) and the English abstract (the logit
// is a sum over 2-D frequency blocks).  For query head g of KV head h:
//   mae_g = (1/T) sum_t | scale q_g.k_t - scale q_g.khat_t |
// where khat_t is the dequantised cached key.  q_g.khat_t is computed in the
// key codec domain, as the decode kernel does: qc_g = (1/sqrt(piece)) H
// (signs * de-whitening * q_g in codec order), and q_g.khat_t = qc_g . y_t with
// y_t,j = rho_t c_w(j)[code_t,j] (the rotation is orthogonal and symmetric).
// One warp handles one token at a time; lane L holds codec coordinates
// 4L..4L+3 (and original dims 4L..4L+3 for the exact logit).
#include <cuda_fp16.h>

#include "bgtq_internal.h"

namespace bgtq {
namespace {

constexpr int kMaeWarps = 4;
constexpr int kMaeTokPerWarp = 64;

struct MaeParams {
    const __half* q;    // [B][H*G][128]
    const __half* k;    // [B][H][t][128]
    const uint8_t* kc;  // K records of the cache
    const float* kn;    // key norms of the cache
    int64_t cap, t;
    CacheMap map;
    int H, G, bk;
    const HeadTab* heads;
    const float* cent;  // [9][256] centroids (fp16-exact values)
    float scale;
    float* out;         // [B][H*G], zeroed by the host, summed into
};

__global__ void __launch_bounds__(kMaeWarps * 32) logit_mae_kernel(MaeParams p) {
    __shared__ float s_qc[8][kD];   // query heads in the key codec domain
    __shared__ float s_q[8][kD];    // query heads as given
    __shared__ uint32_t s_rec[kMaeWarps][32];
    __shared__ float s_sum[kMaeWarps][8];
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int h = blockIdx.y, b = blockIdx.z;
    const int G = p.G;
    const HeadTab* ht = p.heads + h;
    const int n_coded = ht->n_coded;
    const size_t unit = (size_t)b * p.H + h;

    // ---- rotate the query heads (warp w: heads w and w + 4)
    int pl[4], perm[4];
    float f[4], is[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const int j = 4 * lane + i;
        const bool coded = j < n_coded;
        pl[i] = coded ? ht->plog2[j] : 0;
        perm[i] = ht->perm[j];
        f[i] = coded ? ht->sign_k[j] * ht->dewhiten[j] : 0.0f;
        is[i] = coded ? ht->inv_sqrt[j] : 0.0f;
    }
    for (int g = warp; g < 8; g += kMaeWarps) {
        const __half* qg = p.q + ((size_t)b * p.H * G + (size_t)h * G + (g < G ? g : 0)) * kD;
        float x[4];
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            x[i] = g < G ? __half2float(qg[perm[i]]) * f[i] : 0.0f;
            s_q[g][4 * lane + i] = g < G ? __half2float(qg[4 * lane + i]) : 0.0f;
        }
        // blockwise Hadamard: stage hh pairs (j, j + hh) inside pieces larger than hh
#pragma unroll
        for (int hh = 1; hh <= 2; hh <<= 1) {
            float y[4];
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                const float o = x[i ^ hh];
                y[i] = (1 << pl[i]) > hh ? ((i & hh) ? o - x[i] : x[i] + o) : x[i];
            }
#pragma unroll
            for (int i = 0; i < 4; ++i) x[i] = y[i];
        }
#pragma unroll
        for (int hh = 4; hh < kD; hh <<= 1) {
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                const float o = __shfl_xor_sync(0xffffffffu, x[i], hh >> 2);
                if ((1 << pl[i]) > hh) x[i] = ((4 * lane + i) & hh) ? o - x[i] : x[i] + o;
            }
        }
#pragma unroll
        for (int i = 0; i < 4; ++i) s_qc[g][4 * lane + i] = x[i] * is[i];
    }
    // per-lane codec metadata for decoding the K records
    int wd[4], bitpos[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const int j = 4 * lane + i;
        wd[i] = j < n_coded ? ht->width[j] : -1;
        bitpos[i] = ht->pair_bit[(j >> 1) & (kNB - 1)] + ((j & 1) ? (j < n_coded ? ht->width[j] : 0) : 0);
    }
    __syncthreads();

    float acc[8];
#pragma unroll
    for (int g = 0; g < 8; ++g) acc[g] = 0.0f;
    const int64_t t0 = (int64_t)blockIdx.x * (kMaeWarps * kMaeTokPerWarp) + (int64_t)warp * kMaeTokPerWarp;
    const int rec_words = 4 * p.bk;
    for (int it = 0; it < kMaeTokPerWarp; ++it) {
        const int64_t tok = t0 + it;
        if (tok >= p.t) break;
        int64_t sl = p.map.slot(b, h, tok);
        if (sl < 0) sl = 0;  // page index out of range: unspecified result
        const uint32_t* rsrc = reinterpret_cast<const uint32_t*>(p.kc + sl * (16 * p.bk));
        if (lane < rec_words) s_rec[warp][lane] = rsrc[lane];
        const float rho = p.kn[sl];
        const uint2 kr = *(reinterpret_cast<const uint2*>(p.k + (unit * p.t + tok) * kD) + lane);
        __syncwarp();
        float y[4];
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            y[i] = 0.0f;
            if (wd[i] >= 0) {
                const int w = wd[i], bit = bitpos[i];
                const int wi = bit >> 5, sh = bit & 31;
                uint64_t win = s_rec[warp][wi];
                if (wi + 1 < rec_words) win |= (uint64_t)s_rec[warp][wi + 1] << 32;
                const uint32_t code = (uint32_t)(win >> sh) & ((1u << w) - 1u);
                y[i] = debug_in_range(w <= kWMax && code < (1u << w), nullptr) ? rho * p.cent[256 * w + code] : 0.0f;
            }
        }
        const float kx[4] = {__half2float(__ushort_as_half((unsigned short)(kr.x & 0xffffu))),
                             __half2float(__ushort_as_half((unsigned short)(kr.x >> 16))),
                             __half2float(__ushort_as_half((unsigned short)(kr.y & 0xffffu))),
                             __half2float(__ushort_as_half((unsigned short)(kr.y >> 16)))};
#pragma unroll
        for (int g = 0; g < 8; ++g) {
            if (g >= G) break;
            float d = 0.0f;
#pragma unroll
            for (int i = 0; i < 4; ++i) d += s_q[g][4 * lane + i] * kx[i] - s_qc[g][4 * lane + i] * y[i];
#pragma unroll
            for (int o = 16; o >= 1; o >>= 1) d += __shfl_xor_sync(0xffffffffu, d, o);
            acc[g] += fabsf(p.scale * d);
        }
        __syncwarp();
    }
    if (lane == 0) {
#pragma unroll
        for (int g = 0; g < 8; ++g) s_sum[warp][g] = acc[g];
    }
    __syncthreads();
    if (threadIdx.x < G) {
        float sum = 0.0f;
#pragma unroll
        for (int w = 0; w < kMaeWarps; ++w) sum += s_sum[w][threadIdx.x];
        atomicAdd(p.out + unit * G + threadIdx.x, sum / (float)p.t);
    }
}

}  // namespace

cudaError_t launch_logit_mae(const bgtq_plan& pl, cudaStream_t s, const void* q, const void* k, const bgtq_cache& c,
                             int64_t t, int batch, float scale, float* out) {
    MaeParams p;
    p.q = static_cast<const __half*>(q);
    p.k = static_cast<const __half*>(k);
    p.kc = static_cast<const uint8_t*>(c.k_codes);
    p.kn = c.k_norm;
    p.cap = c.capacity;
    p.map = make_cache_map(c, pl.H, batch, nullptr);
    p.t = t;
    p.H = pl.H;
    p.G = pl.G;
    p.bk = pl.bk;
    p.heads = pl.dev.heads;
    p.cent = pl.dev.cent;
    p.scale = scale;
    p.out = out;
    cudaError_t e = cudaMemsetAsync(out, 0, sizeof(float) * (size_t)batch * pl.H * pl.G, s);
    if (e != cudaSuccess) return e;
    const int64_t per_block = kMaeWarps * kMaeTokPerWarp;
    dim3 grid((unsigned)((t + per_block - 1) / per_block), (unsigned)pl.H, (unsigned)batch);
    logit_mae_kernel<<<grid, kMaeWarps * 32, 0, s>>>(p);
    return cudaGetLastError();
}

}  // namespace bgtq
