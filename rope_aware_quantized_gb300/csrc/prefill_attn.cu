// Fused prefill: causal attention over the prompt's fp16 K/V on the tensor
// cores and, in the same launch, the packed K/V records of the prompt.
//
// Method: "RoPE-Aware Bit Allocation for KV-Cache Quantization" — the packed
// cache (review §1 "Packed-Cache") is written when the prompt is prefilled
// and read by every decode step; the prefill itself attends over the prompt
// as given.  Fusing the quantizer into an attention operator is named as
// future work on the LogQuant page (section "중요성 및 주장").
//
// Grid (query blocks of 64 rows, heaviest first; query heads; sequences),
// 4 warps of 16 query rows.  K and V tiles of 64 keys are staged in shared
// memory by cp.async, two stages, 16-byte chunks XOR-swizzled by row so the
// ldmatrix reads hit 8 distinct bank groups.  S = Q K^T and O += P V are
// m16n8k16 fp16 mma with fp32 accumulation (P rounded to fp16); the softmax
// is online, in the log2 domain.  The CTA of the first query head of each KV
// head also encodes the keys and values of its own 64 positions, before it
// attends, with the warp encoder steps of the append kernel (the records are
// bit-identical to an append of the same tokens).
#include <cuda_fp16.h>

#include <cmath>
#include <mutex>

#include "encode.cuh"

namespace bgtq {
namespace {

constexpr int kPfWarps = 4;
constexpr int kPfRows = 64;                 // query rows per CTA (16 per warp)
constexpr int kPfKeys = 64;                 // keys per tile
constexpr int kPfTile = kPfKeys * kD * 2;   // bytes of a 64 x 128 fp16 tile
constexpr int kPfSmem = 5 * kPfTile;        // Q, then K and V of two stages

struct PfParams {
    const __half* q;  // [B][H*G][T][128]
    const __half* k;  // [B][H][T][128]
    const __half* v;
    void* out;        // [B][H*G][T][128], fp16 or fp32
    int out_dtype;
    int T, H, G;
    float scale_log2;
    // the packed records of the prompt
    uint8_t* kc;
    float* kn;
    uint8_t* vc;
    float* vn;
    CacheMap map;
    const HeadTab* heads;
    const float* thr;
    int bk, bv;
    float v_inv_sqrt;
    __half* k_recent;
    int64_t recent;
    int32_t* status;
};

template <bool B>
struct BoolC {
    static constexpr bool value = B;
};

// byte offset of 16-byte chunk c of row r in a swizzled 64 x 256-byte tile
__device__ __forceinline__ uint32_t swz(int r, int c) { return (uint32_t)(r * 256 + ((c ^ (r & 7)) << 4)); }

__device__ __forceinline__ void cp16z(uint32_t dst, const void* src, bool ok) {
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;\n" ::"r"(dst), "l"(src), "r"(ok ? 16 : 0) : "memory");
}
__device__ __forceinline__ void cp_commit() { asm volatile("cp.async.commit_group;\n" ::: "memory"); }
template <int N>
__device__ __forceinline__ void cp_wait() {
    asm volatile("cp.async.wait_group %0;\n" ::"n"(N) : "memory");
}

__device__ __forceinline__ void ldsm4(uint32_t a, uint32_t (&r)[4]) {
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];\n"
                 : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
                 : "r"(a));
}
__device__ __forceinline__ void ldsm4t(uint32_t a, uint32_t (&r)[4]) {
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0,%1,%2,%3}, [%4];\n"
                 : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
                 : "r"(a));
}
// (not volatile: a pure register operation the compiler may schedule freely)
__device__ __forceinline__ void mma_f16(float (&c)[4], const uint32_t (&a)[4], uint32_t b0, uint32_t b1) {
    asm(
        "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, {%0,%1,%2,%3};\n"
        : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
        : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}
__device__ __forceinline__ float ex2(float x) {
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}
__device__ __forceinline__ uint32_t pack_h2(float lo, float hi) {
    const __half2 h = __floats2half2_rn(lo, hi);
    return *reinterpret_cast<const uint32_t*>(&h);
}

// Copy rows [0, 64) of a row-major [.][128] fp16 matrix starting at `src`
// into the swizzled tile at `dst`; rows >= valid are zero-filled.
__device__ __forceinline__ void stage_rows(uint32_t dst, const __half* src, int valid, int tid) {
#pragma unroll
    for (int i = tid; i < kPfKeys * 16; i += kPfWarps * 32) {
        const int r = i >> 4, c = i & 15;
        const bool ok = r < valid;
        cp16z(dst + swz(r, c), ok ? src + (size_t)r * kD + 8 * c : src, ok);
    }
}

// Encode the keys and values of positions [p0, p0 + n) of (b, h): warp w
// takes the token pairs w, w + 4, ...; the steps are the append kernel's.
__device__ void encode_block(const PfParams& p, int b, int h, int p0, int n, const float* s_thr,
                             uint32_t (*s_rec)[8 * kPairMaxW], uint32_t* s_vmask, int warp, int lane) {
    const HeadTab* ht = p.heads + h;
    EncLane ek, ev;
    enc_lane_load(ek, ht, true, p.bv, p.v_inv_sqrt, lane);
    enc_lane_load(ev, ht, false, p.bv, p.v_inv_sqrt, lane);
    const size_t row0 = ((size_t)b * p.H + h) * p.T;
    const size_t unit = (size_t)b * p.H + h;
    for (int pi = warp; 2 * pi < n; pi += kPfWarps) {
        const int pos0 = p0 + 2 * pi;
        const bool has[2] = {true, 2 * pi + 1 < n};
        // ---- keys of the pair
        float x[2][4];
#pragma unroll
        for (int m = 0; m < 2; ++m) {
            const __half* row = p.k + (row0 + pos0 + m) * kD;
#pragma unroll
            for (int k = 0; k < 4; ++k) x[m][k] = has[m] ? __fmul_rn(__half2float(row[ek.src[k]]), ek.wh[k]) : 0.0f;
        }
        for (int k = lane; k < 2 * 8 * kPairMaxW; k += 32) (&s_rec[0][0])[k] = 0;
        __syncwarp();
        int code[2][4];
        float rho[2];
        warp_encode_n<2>(x, ek.sg, ek.pl, ek.is, ek.wd, ek.n_coded, s_thr, code, rho);
#pragma unroll
        for (int m = 0; m < 2; ++m) pack_k_fields(s_rec[m], code[m], ek, lane);
        __syncwarp();
#pragma unroll
        for (int m = 0; m < 2; ++m) {
            if (!has[m]) continue;
            const int pos = pos0 + m;
            const int64_t sl = p.map.slot(b, h, pos);
            if (sl < 0) {
                if (lane == 0 && p.status) atomicOr(p.status, BGTQ_STATUS_PAGE_RANGE);
                continue;
            }
            uint32_t* dst = reinterpret_cast<uint32_t*>(p.kc + sl * (16 * p.bk));
            if (lane < 4 * p.bk) dst[lane] = s_rec[m][lane];
            if (lane == 0) p.kn[sl] = rho[m];
            if (p.recent > 0 && pos >= p.T - p.recent) {
                // fp16 recent-key ring: the key as given, slot pos mod W
                const uint2 nat = *(reinterpret_cast<const uint2*>(p.k + (row0 + pos) * kD) + lane);
                *(reinterpret_cast<uint2*>(p.k_recent + (unit * p.recent + pos % p.recent) * kD) + lane) = nat;
            }
        }
        __syncwarp();
        // ---- values of the pair: one V record
#pragma unroll
        for (int m = 0; m < 2; ++m) {
            uint2 raw = make_uint2(0u, 0u);
            if (has[m]) raw = *(reinterpret_cast<const uint2*>(p.v + (row0 + pos0 + m) * kD) + lane);
            const float2 a = __half22float2(*reinterpret_cast<const __half2*>(&raw.x));
            const float2 c = __half22float2(*reinterpret_cast<const __half2*>(&raw.y));
            x[m][0] = a.x;
            x[m][1] = a.y;
            x[m][2] = c.x;
            x[m][3] = c.y;
        }
        for (int k = lane; k < 8 * kPairMaxW; k += 32) {
            s_rec[2][k] = 0;
            s_vmask[k] = 0;
        }
        __syncwarp();
        warp_encode_n<2>(x, ev.sg, ev.pl, ev.is, ev.wd, kD, s_thr, code, rho);
#pragma unroll
        for (int m = 0; m < 2; ++m)
            if (has[m]) pack_v_fields(s_rec[2], s_vmask, code[m], m, p.bv, lane);
        __syncwarp();
        const int64_t sl0 = p.map.slot(b, h, pos0);
        if (sl0 >= 0) {
            if (lane == 0) {
                p.vn[sl0] = rho[0];
                if (has[1]) p.vn[sl0 + 1] = rho[1];
            }
            uint32_t* vdst = reinterpret_cast<uint32_t*>(p.vc + (sl0 >> 1) * (32 * p.bv));
            for (int k = lane; k < 8 * p.bv; k += 32) {
                if (has[1]) {
                    vdst[k] = s_rec[2][k];
                } else {
                    // a prompt of odd length ends half-way through a pair:
                    // merge without disturbing the other half
                    atomicAnd(vdst + k, ~s_vmask[k]);
                    atomicOr(vdst + k, s_rec[2][k]);
                }
            }
        } else if (lane == 0 && p.status) {
            atomicOr(p.status, BGTQ_STATUS_PAGE_RANGE);
        }
        __syncwarp();
    }
}

__global__ void __launch_bounds__(kPfWarps * 32, 2) prefill_kernel(PfParams p) {
    extern __shared__ __align__(128) uint8_t smem[];
    __shared__ float s_thr[kThrCompact];
    __shared__ uint32_t s_rec[kPfWarps][3][8 * kPairMaxW];
    __shared__ uint32_t s_vmask[kPfWarps][8 * kPairMaxW];
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31, g = lane >> 2, t = lane & 3;
    const int nqb = (p.T + kPfRows - 1) / kPfRows;
    const int qb = nqb - 1 - (int)blockIdx.x;
    const int hq = blockIdx.y, b = blockIdx.z;
    const int h = hq / p.G;
    const int q0 = qb * kPfRows;
    const __half* qsrc = p.q + (((size_t)b * p.H * p.G + hq) * p.T + q0) * kD;
    const __half* ksrc = p.k + ((size_t)b * p.H + h) * p.T * kD;
    const __half* vsrc = p.v + ((size_t)b * p.H + h) * p.T * kD;
    const uint32_t sQ = (uint32_t)__cvta_generic_to_shared(smem);
    const uint32_t sK0 = sQ + kPfTile, sV0 = sQ + 2 * kPfTile;  // stage s: + 2 s kPfTile

    // the query block and the first K/V tile
    stage_rows(sQ, qsrc, min(kPfRows, p.T - q0), tid);
    stage_rows(sK0, ksrc, min(kPfKeys, p.T), tid);
    stage_rows(sV0, vsrc, min(kPfKeys, p.T), tid);
    cp_commit();
    // the first query head of each KV head encodes its block's keys and values
    if (hq % p.G == 0) {
        stage_thresholds(s_thr, p.thr, tid, kPfWarps * 32);
        __syncthreads();
        encode_block(p, b, h, q0, min(kPfRows, p.T - q0), s_thr, s_rec[warp], s_vmask[warp], warp, lane);
    }
    cp_wait<0>();
    __syncthreads();

    // query fragments of the warp's 16 rows (8 k-chunks of 16 dims)
    uint32_t qa[8][4];
#pragma unroll
    for (int c = 0; c < 8; ++c) {
        const int r = 16 * warp + (lane & 7) + ((lane >> 3) & 1) * 8;
        ldsm4(sQ + swz(r, 2 * c + (lane >> 4)), qa[c]);
    }
    const int row_g = q0 + 16 * warp + g;  // rows row_g and row_g + 8
    float m0 = -INFINITY, m1 = -INFINITY, l0 = 0.0f, l1 = 0.0f;
    float acc[16][4];
#pragma unroll
    for (int n = 0; n < 16; ++n) acc[n][0] = acc[n][1] = acc[n][2] = acc[n][3] = 0.0f;

    // one 64-key tile; kEdge: the diagonal tile (causal mask, keys past T)
    auto tile = [&](int j, auto edge_tag) {
        constexpr bool kEdge = decltype(edge_tag)::value;
        const int st = j & 1;
        const uint32_t sK = sK0 + 2 * st * kPfTile, sV = sV0 + 2 * st * kPfTile;
        if (j + 1 <= qb) {
            const uint32_t nK = sK0 + 2 * (st ^ 1) * kPfTile, nV = sV0 + 2 * (st ^ 1) * kPfTile;
            const int k0 = (j + 1) * kPfKeys;
            stage_rows(nK, ksrc + (size_t)k0 * kD, min(kPfKeys, p.T - k0), tid);
            stage_rows(nV, vsrc + (size_t)k0 * kD, min(kPfKeys, p.T - k0), tid);
        }
        cp_commit();
        cp_wait<1>();
        __syncthreads();
        // ---- S = Q K^T for the warp's 16 rows x 64 keys
        float s[8][4];
#pragma unroll
        for (int n = 0; n < 8; ++n) s[n][0] = s[n][1] = s[n][2] = s[n][3] = 0.0f;
#pragma unroll
        for (int c = 0; c < 8; ++c) {
#pragma unroll
            for (int jj = 0; jj < 4; ++jj) {
                uint32_t kb[4];
                const int key = 16 * jj + (lane & 7) + (lane >> 4) * 8;
                ldsm4(sK + swz(key, 2 * c + ((lane >> 3) & 1)), kb);
                mma_f16(s[2 * jj], qa[c], kb[0], kb[1]);
                mma_f16(s[2 * jj + 1], qa[c], kb[2], kb[3]);
            }
        }
        // ---- online softmax (rows g: e = 0, 1; g + 8: e = 2, 3) in the
        // log2 domain: the running maxima m are of scale log2(e) s; the scale
        // is folded into the exponent's fma
        const float cs = p.scale_log2;
        float mx0 = -INFINITY, mx1 = -INFINITY;
#pragma unroll
        for (int n = 0; n < 8; ++n)
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                if (kEdge) {
                    const int key = j * kPfKeys + 8 * n + 2 * t + (e & 1);
                    const int row = row_g + 8 * (e >> 1);
                    if (key > row || key >= p.T) s[n][e] = -INFINITY;
                }
                if (e < 2) mx0 = fmaxf(mx0, s[n][e]);
                else mx1 = fmaxf(mx1, s[n][e]);
            }
        mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, 1));
        mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, 2));
        mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, 1));
        mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, 2));
        const float n0 = fmaxf(m0, mx0 * cs), n1 = fmaxf(m1, mx1 * cs);
        if (__any_sync(0xffffffffu, n0 != m0 || n1 != m1)) {
            // a maximum moved: rescale (exp2(-inf) = 0 on the first tile)
            const float a0 = ex2(m0 - n0), a1 = ex2(m1 - n1);
            l0 *= a0;
            l1 *= a1;
#pragma unroll
            for (int n = 0; n < 16; ++n) {
                acc[n][0] *= a0;
                acc[n][1] *= a0;
                acc[n][2] *= a1;
                acc[n][3] *= a1;
            }
            m0 = n0;
            m1 = n1;
        }
#pragma unroll
        for (int n = 0; n < 8; ++n) {
            s[n][0] = ex2(fmaf(s[n][0], cs, -n0));
            s[n][1] = ex2(fmaf(s[n][1], cs, -n0));
            s[n][2] = ex2(fmaf(s[n][2], cs, -n1));
            s[n][3] = ex2(fmaf(s[n][3], cs, -n1));
            l0 += s[n][0] + s[n][1];
            l1 += s[n][2] + s[n][3];
        }
        // ---- O += P V (4 k-chunks of 16 keys x 16 n-tiles of 8 dims)
#pragma unroll
        for (int kc = 0; kc < 4; ++kc) {
            const uint32_t pa[4] = {pack_h2(s[2 * kc][0], s[2 * kc][1]), pack_h2(s[2 * kc][2], s[2 * kc][3]),
                                    pack_h2(s[2 * kc + 1][0], s[2 * kc + 1][1]),
                                    pack_h2(s[2 * kc + 1][2], s[2 * kc + 1][3])};
            const int key = 16 * kc + (lane & 7) + ((lane >> 3) & 1) * 8;
#pragma unroll
            for (int n2 = 0; n2 < 8; ++n2) {
                uint32_t vb[4];
                ldsm4t(sV + swz(key, 2 * n2 + (lane >> 4)), vb);
                mma_f16(acc[2 * n2], pa, vb[0], vb[1]);
                mma_f16(acc[2 * n2 + 1], pa, vb[2], vb[3]);
            }
        }
        __syncthreads();  // this stage is refilled by the next iteration
    };
    for (int j = 0; j < qb; ++j) tile(j, BoolC<false>{});
    tile(qb, BoolC<true>{});

    // ---- normalise and store rows row_g, row_g + 8 (dims 8 n + 2 t, + 1)
    l0 += __shfl_xor_sync(0xffffffffu, l0, 1);
    l0 += __shfl_xor_sync(0xffffffffu, l0, 2);
    l1 += __shfl_xor_sync(0xffffffffu, l1, 1);
    l1 += __shfl_xor_sync(0xffffffffu, l1, 2);
    const float i0 = 1.0f / l0, i1 = 1.0f / l1;
    const size_t orow0 = ((size_t)b * p.H * p.G + hq) * p.T;
#pragma unroll
    for (int half = 0; half < 2; ++half) {
        const int row = row_g + 8 * half;
        if (row >= p.T) continue;
        const float inv = half ? i1 : i0;
        const size_t o = (orow0 + row) * kD;
#pragma unroll
        for (int n = 0; n < 16; ++n) {
            const float x0 = acc[n][2 * half] * inv, x1 = acc[n][2 * half + 1] * inv;
            const int d = 8 * n + 2 * t;
            if (p.out_dtype) {
                *reinterpret_cast<float2*>(static_cast<float*>(p.out) + o + d) = make_float2(x0, x1);
            } else {
                *reinterpret_cast<__half2*>(static_cast<__half*>(p.out) + o + d) = __floats2half2_rn(x0, x1);
            }
        }
    }
}

}  // namespace

cudaError_t launch_prefill(const bgtq_plan& pl, cudaStream_t s, const void* q, const void* k, const void* v,
                           int batch, int t, const bgtq_cache& c, void* out, int out_dtype, float scale,
                           int32_t* status) {
    static std::mutex mu;
    static bool done[64] = {false};
    int dev = 0;
    cudaGetDevice(&dev);
    if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
    {
        std::lock_guard<std::mutex> lock(mu);
        if (!done[dev]) {
            const cudaError_t e = cudaFuncSetAttribute(prefill_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                                       kPfSmem);
            if (e != cudaSuccess) return e;
            done[dev] = true;
        }
    }
    PfParams p;
    p.q = static_cast<const __half*>(q);
    p.k = static_cast<const __half*>(k);
    p.v = static_cast<const __half*>(v);
    p.out = out;
    p.out_dtype = out_dtype;
    p.T = t;
    p.H = pl.H;
    p.G = pl.G;
    p.scale_log2 = scale * 1.4426950408889634f;
    p.kc = static_cast<uint8_t*>(c.k_codes);
    p.kn = c.k_norm;
    p.vc = static_cast<uint8_t*>(c.v_codes);
    p.vn = c.v_norm;
    p.map = make_cache_map(c, pl.H);
    p.heads = pl.dev.heads;
    p.thr = pl.dev.thr;
    p.bk = pl.bk;
    p.bv = pl.bv;
    p.v_inv_sqrt = (float)(1.0 / std::sqrt((double)kD));
    p.k_recent = static_cast<__half*>(c.k_recent);
    p.recent = c.recent;
    p.status = status;
    dim3 grid((unsigned)((t + kPfRows - 1) / kPfRows), (unsigned)(pl.H * pl.G), (unsigned)batch);
    prefill_kernel<<<grid, kPfWarps * 32, kPfSmem, s>>>(p);
    return cudaGetLastError();
}

}  // namespace bgtq
