// Fused prefill: causal attention over the prompt's fp16 K/V on the
// fifth-generation tensor cores (tcgen05 MMAs with accumulators in tensor
// memory, tiles copied by TMA) and, in the same launch, the packed K/V
// records of the prompt.
//
// Method: "RoPE-Aware Bit Allocation for KV-Cache Quantization" — the packed
// cache (review §1 "Packed-Cache") is written when the prompt is prefilled
// and read by every decode step; the prefill itself attends over the prompt
// as given.  Fusing the quantizer into an attention operator is named as
// future work on the LogQuant page (section "중요성 및 주장").
//
// One CTA takes 128 query rows of two query heads that share a KV head, so
// that both attend the same K/V tiles; 12 warps:
//   warps 0-3, 4-7  softmax warpgroups: thread i of warpgroup g owns row i of
//                   query head g, which is lane i of tensor memory
//   warp 8          issues the MMAs (one thread) and owns the tensor memory
//   warp 9          issues the TMA copies (one thread)
//   warps 10-11     encode the packed records of a share of the block's
//                   positions while the others attend
// Tensor memory, 512 columns of fp32: S_g = Q_g K^T at columns 128 g, the
// output accumulator O_g at 256 + 128 g.  The softmax writes P_g (fp16, two
// per column) over the first 64 columns of S_g and O_g += P_g V reads its A
// operand from there.  Shared memory holds Q_0, Q_1 and two stages of K and
// V tiles (128 x 128 fp16 each), each tile two 64-column TMA boxes with the
// 128-byte swizzle that the MMA descriptors name: Q and K are K-major
// operands, V the MN-major B operand of P V.  MMA order for key tile j:
// PV_0(j), S_0(j+1), PV_1(j), S_1(j+1); warpgroup 0's softmax of a tile runs
// while the tensor cores serve warpgroup 1 and the other way round.  The
// softmax is online in the log2 domain; a row's running maximum is raised
// (and its O rescaled in tensor memory) only when a tile's maximum exceeds
// it by more than kHeadroom, so a probability never exceeds 2^kHeadroom.
// The records of a block's 128 positions are encoded, with the warp encoder
// steps of the append kernel (bit-identical to an append of the same tokens),
// by the encoder warps of the KV head's CTAs of that block, an even share each.
// Every wait is bounded: after kWaitNs it sets BGTQ_STATUS_TIMEOUT, the CTA
// skips the rest of its work, lets its copies and MMAs land and frees its
// tensor memory.
#include <cuda.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>

#include <cmath>
#include <mutex>

#include "prefill_common.cuh"
#include "tc_common.cuh"

namespace bgtq {
namespace {

constexpr int kTcRows = 128;                      // query rows per warpgroup (tensor-memory lanes)
constexpr int kTcKeys = 128;                      // keys per tile
constexpr int kTcThreads = 384;                   // two softmax warpgroups, the MMA warp, the TMA warp, 2 encoder warps
constexpr int kEncWarps = 2;                      // warps that encode records alongside the attention
constexpr int kEncWarp0 = 10;
constexpr uint32_t kTcTile = kTcRows * kD * 2;    // one 128 x 128 fp16 tile: 32 KB
constexpr uint32_t kTcBox = kTcTile / 2;          // one 64-column box of it (128 rows x 128 B)
constexpr uint32_t kOffQ = 0;                     // Q_g at + g kTcTile
constexpr uint32_t kOffK = 2 * kTcTile;           // K stage s at + s kTcTile
constexpr uint32_t kOffV = 4 * kTcTile;           // V stage s at + s kTcTile
constexpr uint32_t kTcSmem = 6 * kTcTile + 1024;  // + room to align the base to 1 KB
constexpr uint32_t kTmemCols = 512;
constexpr float kHeadroom = 8.0f;

// mbarriers: tile copies landed (Q, K/V per stage), stages free again,
// S_g computed, P_g written, O_g final, every MMA done
enum {
    kBarQ = 0,
    kBarKFull = 1,
    kBarVFull = 3,
    kBarKEmpty = 5,
    kBarVEmpty = 7,
    kBarS = 9,
    kBarP = 11,
    kBarO = 13,
    kBarDrain = 15,
    kNumBars = 16
};


// The descriptors the kernel builds, checked field by field for the extreme
// addresses it can use (a 1 KB-aligned base anywhere in the 227 KB a CTA can
// address).
bool descriptors_valid() {
    if (!instr_desc_ok(instr_desc(kTcRows, kTcKeys, 0), 0) || !instr_desc_ok(instr_desc(kTcRows, kD, 1), 1)) return false;
    constexpr uint32_t kMaxSmem = 227u * 1024u;
    for (uint32_t base = 0; base + kTcSmem <= kMaxSmem + 1024; base += 1024)
        for (int k = 0; k < kD / 16; ++k) {
            // S operands (K-major: LBO unused, SBO = 8 rows of 128 B), steps of 16 in K
            const uint32_t off = (uint32_t)(k >> 2) * kTcBox + (uint32_t)(k & 3) * 32;
            if (!smem_desc_ok(base + kOffQ + kTcTile + off, 16, 1024) || !smem_desc_ok(base + kOffK + kTcTile + off, 16, 1024))
                return false;
            // V (MN-major: LBO = the 64-column box stride, SBO = 8 keys of 128 B), steps of 16 keys
            if (!smem_desc_ok(base + kOffV + kTcTile + (uint32_t)k * 2048, kTcBox, 1024)) return false;
        }
    return true;
}

// Softmax warpgroup g: the online softmax of row r of query head hq0 + g
// over key tiles 0 .. nkt-1, then the normalised output row.
__device__ __forceinline__ void softmax_rows(const PfParams& p, uint32_t tmem, int g, int b, int hq, int q0, int nkt,
                                             uint32_t bar_s, uint32_t bar_p, uint32_t bar_o, volatile int* abort_flag,
                                             int warp, int lane) {
    const int r = 32 * (warp & 3) + lane;  // row of the block = tensor-memory lane
    const int row = q0 + r;
    const uint32_t lanes = (uint32_t)(32 * (warp & 3)) << 16;
    const uint32_t tS = tmem + lanes + 128u * g, tO = tmem + lanes + 256u + 128u * g;
    const float c = p.scale_log2;
    float m = 0.0f, l = 0.0f;
    bool ok = true;
    for (int j = 0; j < nkt; ++j) {
        if (!__all_sync(0xffffffffu, mbar_wait(bar_s, j & 1, abort_flag, p.status))) {
            ok = false;
            break;
        }
        tc_fence_after();
        float s[kTcKeys];
#pragma unroll
        for (int q = 0; q < kTcKeys / 32; ++q) tmem_ld32(tS + 32 * q, s + 32 * q);
#pragma unroll
        for (int q = 0; q < kTcKeys / 32; ++q) tmem_wait_ld32(s + 32 * q);
        if (j == nkt - 1) {  // the diagonal tile: keys after the row, and past the prompt
            const int lim = min(row, p.T - 1) - j * kTcKeys;
#pragma unroll
            for (int k = 0; k < kTcKeys; ++k)
                if (k > lim) s[k] = -INFINITY;
        }
        float mx[8];
#pragma unroll
        for (int i = 0; i < 8; ++i) mx[i] = s[i];
#pragma unroll
        for (int k = 8; k < kTcKeys; ++k) mx[k & 7] = fmaxf(mx[k & 7], s[k]);
        const float mt = fmaxf(fmaxf(fmaxf(mx[0], mx[1]), fmaxf(mx[2], mx[3])),
                               fmaxf(fmaxf(mx[4], mx[5]), fmaxf(mx[6], mx[7]))) * c;
        float f = 1.0f;
        bool raise = false;
        if (j == 0) {
            m = mt;  // key 0 is before every row: finite
        } else if (mt > m + kHeadroom) {
            f = ex2(m - mt);
            m = mt;
            l *= f;
            raise = true;
        }
        if (__any_sync(0xffffffffu, raise)) {
            // the row's O so far is in tensor memory; PV of tile j-1 has
            // completed (S of tile j was issued after it)
#pragma unroll 1
            for (int q = 0; q < kD / 32; ++q) {
                float o[32];
                tmem_ld32(tO + 32 * q, o);
                tmem_wait_ld32(o);
                uint32_t w[32];
#pragma unroll
                for (int i = 0; i < 32; ++i) w[i] = __float_as_uint(o[i] * f);
                tmem_st32(tO + 32 * q, w);
            }
        }
        uint32_t pk[kTcKeys / 2];
        float ls[4] = {0.0f, 0.0f, 0.0f, 0.0f};
#pragma unroll
        for (int i = 0; i < kTcKeys / 2; ++i) {
            const float p0 = ex2(fmaf(s[2 * i], c, -m)), p1 = ex2(fmaf(s[2 * i + 1], c, -m));
            ls[i & 3] += p0 + p1;
            pk[i] = pack_h2(p0, p1);
        }
        l += (ls[0] + ls[1]) + (ls[2] + ls[3]);
        // P over the first 64 columns of S (already read)
        tmem_st32(tS, pk);
        tmem_st32(tS + 32, pk + 32);
        tmem_wait_st();
        tc_fence_before();
        mbar_arrive(bar_p);
    }
    if (!ok || !__all_sync(0xffffffffu, mbar_wait(bar_o, 0, abort_flag, p.status))) return;
    tc_fence_after();
    const float inv = 1.0f / l;
    const size_t o0 = ((size_t)((size_t)b * p.H * p.G + hq) * p.T + row) * kD;
#pragma unroll 1
    for (int q = 0; q < kD / 32; ++q) {
        float o[32];
        tmem_ld32(tO + 32 * q, o);
        tmem_wait_ld32(o);
        if (row >= p.T) continue;
        if (p.out_dtype) {
            float4* dst = reinterpret_cast<float4*>(static_cast<float*>(p.out) + o0 + 32 * q);
#pragma unroll
            for (int i = 0; i < 8; ++i)
                dst[i] = make_float4(o[4 * i] * inv, o[4 * i + 1] * inv, o[4 * i + 2] * inv, o[4 * i + 3] * inv);
        } else {
            uint4* dst = reinterpret_cast<uint4*>(static_cast<__half*>(p.out) + o0 + 32 * q);
#pragma unroll
            for (int i = 0; i < 4; ++i)
                dst[i] = make_uint4(pack_h2(o[8 * i] * inv, o[8 * i + 1] * inv), pack_h2(o[8 * i + 2] * inv, o[8 * i + 3] * inv),
                                    pack_h2(o[8 * i + 4] * inv, o[8 * i + 5] * inv),
                                    pack_h2(o[8 * i + 6] * inv, o[8 * i + 7] * inv));
        }
    }
}

__global__ void __launch_bounds__(kTcThreads, 1)
    prefill_kernel(const __grid_constant__ CUtensorMap tq, const __grid_constant__ CUtensorMap tk,
                   const __grid_constant__ CUtensorMap tv, PfParams p) {
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    __shared__ __align__(8) uint64_t s_bar[kNumBars];
    __shared__ uint32_t s_tmem;
    __shared__ int s_abort;
    __shared__ float s_thr[kThrCompact];
    __shared__ uint32_t s_rec[kEncWarps][3][8 * kPairMaxW];
    __shared__ uint32_t s_vmask[kEncWarps][8 * kPairMaxW];
    const uint32_t sbase = (smem_u32(smem_raw) + 1023u) & ~1023u;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int npair = (p.G + 1) >> 1;
    const int pair = (int)blockIdx.x % npair;
    const int h = (int)(blockIdx.x / npair) % p.H;
    const int b = (int)blockIdx.x / (npair * p.H);
    const int nqb = (p.T + kTcRows - 1) / kTcRows;
    const int qb = nqb - 1 - (int)blockIdx.y;  // heaviest query blocks first
    const int q0 = qb * kTcRows;
    const int hq0 = h * p.G + 2 * pair;
    const int ng = 2 * pair + 1 < p.G ? 2 : 1;  // query heads of this CTA
    const int nkt = qb + 1;                     // key tiles; tile qb holds the diagonal
    const uint32_t bar0 = smem_u32(&s_bar[0]);
    volatile int* abort_flag = &s_abort;
#define BAR(i) (bar0 + 8u * (uint32_t)(i))

    if (tid == 0) {
        s_abort = 0;
        for (int i = 0; i < kNumBars; ++i) mbar_init(BAR(i), (i == kBarP || i == kBarP + 1) ? kTcRows : 1);
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    if (warp == 8) {
        asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(&s_tmem)),
                     "r"(kTmemCols));
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;");
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = s_tmem;

    if (warp == 9) {
        // ---- TMA: Q of the CTA's heads, then K and V tiles through two stages
        if (lane == 0) {
            int used[2] = {0, 0};
            const int qrow = ((b * p.H * p.G) + hq0) * p.T + q0;
            mbar_expect_tx(BAR(kBarQ), ng * kTcTile);
            for (int g = 0; g < ng; ++g)
                for (int x = 0; x < 2; ++x)
                    tma_load_2d(sbase + kOffQ + g * kTcTile + x * kTcBox, &tq, 64 * x, qrow + g * p.T, BAR(kBarQ));
            const int krow = (b * p.H + h) * p.T;
            for (int j = 0; j < nkt; ++j) {
                const int s = j & 1;
                const uint32_t par = (uint32_t)((j >> 1) - 1) & 1u;
                if (j >= 2 && !mbar_wait(BAR(kBarKEmpty + s), par, abort_flag, p.status)) break;
                mbar_expect_tx(BAR(kBarKFull + s), kTcTile);
                for (int x = 0; x < 2; ++x)
                    tma_load_2d(sbase + kOffK + s * kTcTile + x * kTcBox, &tk, 64 * x, krow + j * kTcKeys, BAR(kBarKFull + s));
                if (j >= 2 && !mbar_wait(BAR(kBarVEmpty + s), par, abort_flag, p.status)) {
                    used[s] = 2 * j + 1;  // K of tile j in flight, V not
                    break;
                }
                mbar_expect_tx(BAR(kBarVFull + s), kTcTile);
                for (int x = 0; x < 2; ++x)
                    tma_load_2d(sbase + kOffV + s * kTcTile + x * kTcBox, &tv, 64 * x, krow + j * kTcKeys, BAR(kBarVFull + s));
                used[s] = 2 * j + 2;
            }
            // every copy issued has landed before the CTA ends (normally at
            // once: the MMA thread waited for them)
            mbar_wait(BAR(kBarQ), 0, abort_flag, p.status, false);
            for (int s = 0; s < 2; ++s) {
                if (used[s] == 0) continue;
                const int jl = (used[s] - 1) >> 1;  // last tile on this stage
                const uint32_t par = (uint32_t)(jl >> 1) & 1u;
                mbar_wait(BAR(kBarKFull + s), par, abort_flag, p.status, false);
                if (used[s] & 1) {  // its V was not issued: the previous use's V
                    if (jl >= 2) mbar_wait(BAR(kBarVFull + s), par ^ 1u, abort_flag, p.status, false);
                } else {
                    mbar_wait(BAR(kBarVFull + s), par, abort_flag, p.status, false);
                }
            }
        }
        __syncwarp();
    } else if (warp == 8) {
        // ---- MMA issue
        if (lane == 0) {
            constexpr uint32_t idS = instr_desc(kTcRows, kTcKeys, 0);
            constexpr uint32_t idO = instr_desc(kTcRows, kD, 1);
            auto issue_s = [&](int g, int j) {
                const uint32_t qa = sbase + kOffQ + g * kTcTile, ka = sbase + kOffK + (j & 1) * kTcTile;
#pragma unroll
                for (int k = 0; k < kD / 16; ++k) {
                    const uint32_t off = (uint32_t)(k >> 2) * kTcBox + (uint32_t)(k & 3) * 32;
                    mma_ss(tmem + 128u * g, smem_desc(qa + off, 16, 1024), smem_desc(ka + off, 16, 1024), idS, k > 0);
                }
                mma_commit(BAR(kBarS + g));
            };
            auto issue_pv = [&](int g, int j) {
                const uint32_t va = sbase + kOffV + (j & 1) * kTcTile;
#pragma unroll
                for (int k = 0; k < kTcKeys / 16; ++k)
                    mma_ts(tmem + 256u + 128u * g, tmem + 128u * g + 8u * k, smem_desc(va + 2048u * k, kTcBox, 1024), idO,
                           (j > 0 || k > 0) ? 1u : 0u);
            };
            bool ok = mbar_wait(BAR(kBarQ), 0, abort_flag, p.status) && mbar_wait(BAR(kBarKFull), 0, abort_flag, p.status);
            if (ok) {
                tc_fence_after();
                for (int g = 0; g < ng; ++g) issue_s(g, 0);
                mma_commit(BAR(kBarKEmpty));
            }
            for (int j = 0; ok && j < nkt; ++j) {
                const int s = j & 1;
                const bool next = j + 1 < nkt;
                if (!mbar_wait(BAR(kBarVFull + s), (uint32_t)(j >> 1) & 1u, abort_flag, p.status)) break;
                for (int g = 0; g < ng && ok; ++g) {
                    ok = mbar_wait(BAR(kBarP + g), (uint32_t)j & 1u, abort_flag, p.status);
                    if (ok && next && g == 0)
                        ok = mbar_wait(BAR(kBarKFull + (s ^ 1)), (uint32_t)((j + 1) >> 1) & 1u, abort_flag, p.status);
                    if (!ok) break;
                    tc_fence_after();
                    issue_pv(g, j);
                    if (next) {
                        issue_s(g, j + 1);
                    } else {
                        mma_commit(BAR(kBarO + g));
                    }
                }
                if (!ok) break;
                mma_commit(BAR(kBarVEmpty + s));
                if (next) mma_commit(BAR(kBarKEmpty + (s ^ 1)));
            }
            // every MMA issued has completed before the CTA ends
            mma_commit(BAR(kBarDrain));
            mbar_wait(BAR(kBarDrain), 0, abort_flag, p.status, false);
        }
        __syncwarp();
    } else if (warp >= kEncWarp0) {
        // ---- record encoder: the block's 128 positions are shared out over
        // the CTAs of the KV head's query-head pairs (an even share each, so a
        // V pair record is never split); encoded while the others attend
        const int n = min(kTcRows, p.T - q0);
        const int share = ((n + npair - 1) / npair + 1) & ~1;
        const int e0 = pair * share, e1 = min(n, e0 + share);
        if (e0 < e1) {
            const int ew = warp - kEncWarp0;
            stage_thresholds(s_thr, p.thr, tid - kEncWarp0 * 32, kEncWarps * 32);
            asm volatile("bar.sync 1, %0;" ::"n"(kEncWarps * 32) : "memory");
            encode_block(p, b, h, q0 + e0, e1 - e0, 0, p.T, s_thr, s_rec[ew], s_vmask[ew], ew, lane, kEncWarps);
        }
    } else {
        // ---- softmax warpgroups
        const int g = warp >> 2;
        if (g < ng)
            softmax_rows(p, tmem, g, b, hq0 + g, q0, nkt, BAR(kBarS + g), BAR(kBarP + g), BAR(kBarO + g), abort_flag, warp,
                         lane);
    }
#undef BAR
    tc_fence_before();
    __syncthreads();
    if (warp == 8) {
        tc_fence_after();
        asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(kTmemCols));
    }
}

}  // namespace

cudaError_t launch_prefill(const bgtq_plan& pl, cudaStream_t s, const void* q, const void* k, const void* v,
                           int batch, int t, const bgtq_cache& c, void* out, int out_dtype, float scale,
                           int32_t* status) {
    static std::mutex mu;
    static bool done[64] = {false};
    static const bool desc_ok = descriptors_valid();
    if (!desc_ok) return cudaErrorInvalidValue;
    // coordinates of the tensor maps and the grid are 32-bit
    const uint64_t q_rows = (uint64_t)batch * pl.H * pl.G * (uint64_t)t;
    const int nqb = (t + kTcRows - 1) / kTcRows;
    const uint64_t units = (uint64_t)batch * pl.H * ((pl.G + 1) / 2);
    if (q_rows + kTcRows >= (1ull << 31) || nqb > 65535 || units >= (1ull << 31)) return cudaErrorInvalidValue;
    int dev = 0;
    cudaGetDevice(&dev);
    if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
    {
        std::lock_guard<std::mutex> lock(mu);
        if (!done[dev]) {
            const cudaError_t e =
                cudaFuncSetAttribute(prefill_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kTcSmem);
            if (e != cudaSuccess) return e;
            done[dev] = true;
        }
    }
    alignas(64) CUtensorMap tq, tk, tv;
    if (!rows_map(&tq, q, q_rows, kTcRows) || !rows_map(&tk, k, (uint64_t)batch * pl.H * t, kTcKeys) ||
        !rows_map(&tv, v, (uint64_t)batch * pl.H * t, kTcKeys))
        return cudaErrorInvalidValue;
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
    p.map = make_cache_map(c, pl.H, batch, status);
    p.heads = pl.dev.heads;
    p.thr = pl.dev.thr;
    p.bk = pl.bk;
    p.bv = pl.bv;
    p.v_inv_sqrt = (float)(1.0 / std::sqrt((double)kD));
    p.k_recent = static_cast<__half*>(c.k_recent);
    p.recent = c.recent;
    p.status = status;
    const dim3 grid((unsigned)units, (unsigned)nqb, 1);
    prefill_kernel<<<grid, kTcThreads, kTcSmem, s>>>(tq, tk, tv, p);
    return cudaGetLastError();
}

}  // namespace bgtq
