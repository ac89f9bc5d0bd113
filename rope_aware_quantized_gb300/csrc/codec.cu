// TQ-MSE encoder (quantize-append) and decoder (debug dequant) for the
// Block-GTQ packed cache.
//
// Method: "RoPE-Aware Bit Allocation for KV-Cache Quantization" — review §1
// Key Terms (TQ-MSE rotates then quantises; the packed cache stores
// compressed K/V) and English abstract (per-block integer widths for keys,
// uniform TQ-MSE for values).  One warp encodes one token: lane L holds codec
// coordinates 4L..4L+3.  Every float operation is a single correctly rounded
// IEEE operation in a fixed order (this file is built with --fmad=false and
// uses explicit _rn intrinsics), so codes, norms and decoded values are
// bit-identical to any implementation that follows the same steps.
#include <cuda_fp16.h>

#include "bgtq_internal.h"

namespace bgtq {
namespace {

constexpr int kWarpsQ = 4;
constexpr int kPairsPerWarp = 8;  // token pairs each warp of quantize_append encodes

struct QParams {
    const __half* k;
    const __half* v;
    int t_new, H;
    const int32_t* pos_start;
    uint8_t* kc;
    float* kn;
    uint8_t* vc;
    float* vn;
    int64_t cap;
    const HeadTab* heads;
    const float* thr;
    int bk, bv;
    float v_inv_sqrt;
    int32_t* status;
};

// Randomized Hadamard on the warp's 128 slots: stages h = 1, 2, 4, ..., 64,
// pair (j, j+h) inside a piece larger than h becomes (a + b, a - b).
__device__ __forceinline__ void warp_butterflies(float (&x)[4], const int (&plog2)[4], int lane) {
#pragma unroll
    for (int h = 1; h <= 2; h <<= 1) {
        float y[4];
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const int partner = i ^ h;
            const bool active = (1 << plog2[i]) > h;
            y[i] = !active ? x[i] : ((i & h) ? __fsub_rn(x[partner], x[i]) : __fadd_rn(x[i], x[partner]));
        }
#pragma unroll
        for (int i = 0; i < 4; ++i) x[i] = y[i];
    }
#pragma unroll
    for (int h = 4; h < 128; h <<= 1) {
        const int lm = h >> 2;
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const float other = __shfl_xor_sync(0xffffffffu, x[i], lm);
            const int j = 4 * lane + i;
            if ((1 << plog2[i]) > h) x[i] = (j & h) ? __fsub_rn(other, x[i]) : __fadd_rn(x[i], other);
        }
    }
}

// Encode one token held as x[4] per lane (already whitened for keys).
// Returns the codes of the lane's four coordinates and the norm rho.
__device__ __forceinline__ float warp_encode(float (&x)[4], const float (&sgn)[4], const int (&plog2)[4],
                                             const float (&inv_sqrt)[4], const int (&width)[4], int n_coded,
                                             const float* __restrict__ thr, int lane, int (&code)[4]) {
#pragma unroll
    for (int i = 0; i < 4; ++i) x[i] = __fmul_rn(x[i], sgn[i]);
    warp_butterflies(x, plog2, lane);
#pragma unroll
    for (int i = 0; i < 4; ++i) x[i] = __fmul_rn(x[i], inv_sqrt[i]);
    float part = __fadd_rn(__fadd_rn(__fmul_rn(x[0], x[0]), __fmul_rn(x[1], x[1])),
                           __fadd_rn(__fmul_rn(x[2], x[2]), __fmul_rn(x[3], x[3])));
#pragma unroll
    for (int m = 16; m >= 1; m >>= 1) part = __fadd_rn(part, __shfl_xor_sync(0xffffffffu, part, m));
    const float rho = __fsqrt_rn(__fdiv_rn(part, (float)n_coded));
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const float u = rho > 0.0f ? __fdiv_rn(x[i], rho) : 0.0f;
        const int n = 1 << width[i];
        const float* tb = thr + 256 * width[i];
        int pos = 0;
#pragma unroll
        for (int s = 128; s >= 1; s >>= 1) {
            if (2 * s <= n) {
                if (tb[pos + s - 1] <= u) pos += s;
            }
        }
        code[i] = pos;
    }
    return rho;
}

__global__ void __launch_bounds__(128) quantize_append_kernel(QParams p) {
    __shared__ __align__(16) float s_thr[(kWMax + 1) * 256];
    __shared__ float xs[kWarpsQ][kD];
    __shared__ uint32_t krec[kWarpsQ][32];
    __shared__ uint32_t vrec[kWarpsQ][8 * kPairMaxW];
    __shared__ uint32_t vmask[kWarpsQ][8 * kPairMaxW];
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int h = blockIdx.y, b = blockIdx.z;
    // The next kernel may launch right away (programmatic dependent launch);
    // the plan's tables are static, the inputs are read after the wait.
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
    // Lloyd-Max thresholds of every width, staged once per block
    for (int i = threadIdx.x; i < (kWMax + 1) * 256 / 4; i += kWarpsQ * 32)
        reinterpret_cast<float4*>(s_thr)[i] = __ldg(reinterpret_cast<const float4*>(p.thr) + i);
    __syncthreads();
    asm volatile("griddepcontrol.wait;" ::: "memory");
    const int ps = p.pos_start[b];
    if (ps < 0 || (int64_t)ps + p.t_new > p.cap) {
        if (blockIdx.x == 0 && h == 0 && threadIdx.x == 0 && p.status) atomicOr(p.status, BGTQ_STATUS_APPEND_CAPACITY);
        return;
    }
    const HeadTab* ht = p.heads + h;
    const int n_coded = ht->n_coded;
    const size_t unit = (size_t)b * p.H + h;
    const int krec_words = 4 * p.bk, vrec_words = 8 * p.bv;

    // per-lane key codec metadata (codec coordinates 4*lane + i)
    int kpl[4], kw[4], kperm[4];
    float ksg[4], kis[4], kwh[4];
    int vpl[4], vw[4];
    float vsg[4], vis[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const int j = 4 * lane + i;
        const bool coded = j < n_coded;
        kpl[i] = coded ? ht->plog2[j] : 0;
        kw[i] = coded ? ht->width[j] : 0;
        kperm[i] = ht->perm[j];
        ksg[i] = ht->sign_k[j];
        kis[i] = ht->inv_sqrt[j];
        kwh[i] = ht->whiten[j];
        vpl[i] = 7;
        vw[i] = p.bv;
        vsg[i] = ht->sign_v[j];
        vis[i] = p.v_inv_sqrt;
    }
    const int64_t P_first = (int64_t)(ps >> 1) + ((int64_t)blockIdx.x * kWarpsQ + warp) * kPairsPerWarp;
    for (int it = 0; it < kPairsPerWarp; ++it) {
        const int64_t P = P_first + it;  // token-pair index
        const int64_t pos0 = 2 * P;
        const bool has[2] = {pos0 >= ps && pos0 < (int64_t)ps + p.t_new, pos0 + 1 >= ps && pos0 + 1 < (int64_t)ps + p.t_new};
        if (!has[0] && !has[1]) continue;
        for (int i = lane; i < 8 * kPairMaxW; i += 32) {
            vrec[warp][i] = 0;
            vmask[warp][i] = 0;
        }
        for (int par = 0; par < 2; ++par) {
            if (!has[par]) continue;
            const int64_t pos = pos0 + par;
            const size_t tok = (size_t)(pos - ps);
            // ---- key
            {
                const __half2* src = reinterpret_cast<const __half2*>(p.k + (unit * p.t_new + tok) * kD) + 2 * lane;
                const float2 a = __half22float2(src[0]), c = __half22float2(src[1]);
                xs[warp][4 * lane + 0] = a.x;
                xs[warp][4 * lane + 1] = a.y;
                xs[warp][4 * lane + 2] = c.x;
                xs[warp][4 * lane + 3] = c.y;
                if (lane < 32) krec[warp][lane] = 0;
                __syncwarp();
                float x[4];
#pragma unroll
                for (int i = 0; i < 4; ++i) x[i] = (4 * lane + i < n_coded) ? __fmul_rn(xs[warp][kperm[i]], kwh[i]) : 0.0f;
                int code[4];
                const float rho = warp_encode(x, ksg, kpl, kis, kw, n_coded, s_thr, lane, code);
#pragma unroll
                for (int pr = 0; pr < 2; ++pr) {
                    const int j = 4 * lane + 2 * pr;
                    if (j + 1 < n_coded) {
                        const int w = kw[2 * pr];
                        const uint32_t field = (uint32_t)code[2 * pr] | ((uint32_t)code[2 * pr + 1] << w);
                        const int bit = ht->pair_bit[j >> 1];
                        const int wi = bit >> 5, sh = bit & 31;
                        atomicOr(&krec[warp][wi], field << sh);
                        if (sh + 2 * w > 32) atomicOr(&krec[warp][wi + 1], field >> (32 - sh));
                    }
                }
                __syncwarp();
                uint32_t* dst = reinterpret_cast<uint32_t*>(p.kc + (unit * p.cap + pos) * (16 * p.bk));
                if (lane < krec_words) dst[lane] = krec[warp][lane];
                if (lane == 0) p.kn[unit * p.cap + pos] = rho;
                __syncwarp();
            }
            // ---- value
            {
                const __half2* src = reinterpret_cast<const __half2*>(p.v + (unit * p.t_new + tok) * kD) + 2 * lane;
                const float2 a = __half22float2(src[0]), c = __half22float2(src[1]);
                float x[4] = {a.x, a.y, c.x, c.y};
                int code[4];
                const float rho = warp_encode(x, vsg, vpl, vis, vw, kD, s_thr, lane, code);
                const uint32_t m1 = (1u << p.bv) - 1;
#pragma unroll
                for (int i = 0; i < 4; ++i) {
                    const int j = 4 * lane + i;
                    const int bit = 2 * p.bv * j + par * p.bv;
                    const int wi = bit >> 5, sh = bit & 31;
                    atomicOr(&vrec[warp][wi], (uint32_t)code[i] << sh);
                    atomicOr(&vmask[warp][wi], m1 << sh);
                    if (sh + p.bv > 32) {
                        atomicOr(&vrec[warp][wi + 1], (uint32_t)code[i] >> (32 - sh));
                        atomicOr(&vmask[warp][wi + 1], m1 >> (32 - sh));
                    }
                }
                if (lane == 0) p.vn[unit * p.cap + pos] = rho;
            }
        }
        __syncwarp();
        uint32_t* vdst = reinterpret_cast<uint32_t*>(p.vc + (unit * (p.cap / 2) + P) * (32 * p.bv));
        for (int i = lane; i < vrec_words; i += 32) {
            uint32_t val = vrec[warp][i];
            if (!(has[0] && has[1])) val = (vdst[i] & ~vmask[warp][i]) | val;
            vdst[i] = val;
        }
        __syncwarp();
    }
}

struct DqParams {
    const uint8_t* kc;
    const float* kn;
    const uint8_t* vc;
    const float* vn;
    int64_t cap, t0, t1;
    size_t unit;
    const HeadTab* ht;
    const float* cent;
    int bk, bv;
    float v_inv_sqrt;
    float* k_out;
    float* v_out;
    int codec_domain;
};

__global__ void __launch_bounds__(128) dequant_kernel(DqParams p) {
    __shared__ uint32_t rec[kWarpsQ][8 * kPairMaxW];
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int64_t t = p.t0 + (int64_t)blockIdx.x * kWarpsQ + warp;
    if (t >= p.t1) return;
    const HeadTab* ht = p.ht;
    const int64_t row = t - p.t0;
    if (p.k_out) {
        const uint32_t* src = reinterpret_cast<const uint32_t*>(p.kc + (p.unit * p.cap + t) * (16 * p.bk));
        if (lane < 4 * p.bk) rec[warp][lane] = src[lane];
        __syncwarp();
        const float rho = p.kn[p.unit * p.cap + t];
        const int n_coded = ht->n_coded;
        float y[4];
        int pl[4];
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const int j = 4 * lane + i;
            y[i] = 0.0f;
            pl[i] = 0;
            if (j < n_coded) {
                const int w = ht->width[j];
                const int bit = ht->pair_bit[j >> 1];
                const int wi = bit >> 5, sh = bit & 31;
                uint64_t win = ((uint64_t)rec[warp][wi + 1 < 32 ? wi + 1 : wi] << 32) | rec[warp][wi];
                if (wi + 1 >= 4 * p.bk) win &= 0xffffffffull;
                const uint32_t field = (uint32_t)(win >> sh) & ((1u << (2 * w)) - 1);
                const uint32_t c = (j & 1) ? (field >> w) : (field & ((1u << w) - 1));
                y[i] = __fmul_rn(rho, p.cent[256 * w + c]);
                pl[i] = ht->plog2[j];
            }
        }
        float* out = p.k_out + row * kD;
        if (p.codec_domain) {
#pragma unroll
            for (int i = 0; i < 4; ++i) out[4 * lane + i] = y[i];
        } else {
            warp_butterflies(y, pl, lane);
#pragma unroll
            for (int i = 0; i < 4; ++i) out[4 * lane + i] = 0.0f;
            __syncwarp();
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                const int j = 4 * lane + i;
                if (j < n_coded) {
                    float v = __fmul_rn(y[i], ht->inv_sqrt[j]);
                    v = __fmul_rn(v, ht->sign_k[j]);
                    v = __fmul_rn(v, ht->dewhiten[j]);
                    out[ht->perm[j]] = v;
                }
            }
        }
        __syncwarp();
    }
    if (p.v_out) {
        const uint32_t* src = reinterpret_cast<const uint32_t*>(p.vc + (p.unit * (p.cap / 2) + (t >> 1)) * (32 * p.bv));
        for (int i = lane; i < 8 * p.bv; i += 32) rec[warp][i] = src[i];
        __syncwarp();
        const float rho = p.vn[p.unit * p.cap + t];
        const int par = (int)(t & 1);
        float y[4];
        int pl[4];
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const int j = 4 * lane + i;
            const int bit = 2 * p.bv * j + par * p.bv;
            const int wi = bit >> 5, sh = bit & 31;
            uint64_t win = rec[warp][wi];
            if (wi + 1 < 8 * p.bv) win |= (uint64_t)rec[warp][wi + 1] << 32;
            const uint32_t c = (uint32_t)(win >> sh) & ((1u << p.bv) - 1);
            y[i] = __fmul_rn(rho, p.cent[256 * p.bv + c]);
            pl[i] = 7;
        }
        float* out = p.v_out + row * kD;
        if (p.codec_domain) {
#pragma unroll
            for (int i = 0; i < 4; ++i) out[4 * lane + i] = y[i];
        } else {
            warp_butterflies(y, pl, lane);
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                const int j = 4 * lane + i;
                float v = __fmul_rn(y[i], p.v_inv_sqrt);
                v = __fmul_rn(v, ht->sign_v[j]);
                out[j] = v;
            }
        }
    }
}

}  // namespace

cudaError_t launch_quantize_append(const bgtq_plan& pl, cudaStream_t s, const void* k, const void* v, int batch,
                                   int t_new, const int32_t* pos_start, const bgtq_cache& c, int32_t* status) {
    QParams p;
    p.k = static_cast<const __half*>(k);
    p.v = static_cast<const __half*>(v);
    p.t_new = t_new;
    p.H = pl.H;
    p.pos_start = pos_start;
    p.kc = static_cast<uint8_t*>(c.k_codes);
    p.kn = c.k_norm;
    p.vc = static_cast<uint8_t*>(c.v_codes);
    p.vn = c.v_norm;
    p.cap = c.capacity;
    p.heads = pl.dev.heads;
    p.thr = pl.dev.thr;
    p.bk = pl.bk;
    p.bv = pl.bv;
    p.v_inv_sqrt = (float)(1.0 / std::sqrt((double)kD));
    p.status = status;
    const int64_t pairs = (int64_t)t_new / 2 + 1;
    const int64_t per_block = (int64_t)kWarpsQ * kPairsPerWarp;
    dim3 grid((unsigned)((pairs + per_block - 1) / per_block), (unsigned)pl.H, (unsigned)batch);
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = dim3(32 * kWarpsQ, 1, 1);
    cfg.stream = s;
    cudaLaunchAttribute attr;
    attr.id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr.val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = &attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, quantize_append_kernel, p);
}

cudaError_t launch_dequant(const bgtq_plan& pl, cudaStream_t s, const bgtq_cache& c, int batch, int b, int head,
                           int64_t t0, int64_t t1, float* k_out, float* v_out, int codec_domain) {
    (void)batch;
    DqParams p;
    p.kc = static_cast<const uint8_t*>(c.k_codes);
    p.kn = c.k_norm;
    p.vc = static_cast<const uint8_t*>(c.v_codes);
    p.vn = c.v_norm;
    p.cap = c.capacity;
    p.t0 = t0;
    p.t1 = t1;
    p.unit = (size_t)b * pl.H + head;
    p.ht = pl.dev.heads + head;
    p.cent = pl.dev.cent;
    p.bk = pl.bk;
    p.bv = pl.bv;
    p.v_inv_sqrt = (float)(1.0 / std::sqrt((double)kD));
    p.k_out = k_out;
    p.v_out = v_out;
    p.codec_domain = codec_domain;
    const int64_t n = t1 - t0;
    dequant_kernel<<<(unsigned)((n + kWarpsQ - 1) / kWarpsQ), 32 * kWarpsQ, 0, s>>>(p);
    return cudaGetLastError();
}

}  // namespace bgtq
