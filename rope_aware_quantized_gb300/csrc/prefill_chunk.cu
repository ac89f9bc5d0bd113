// Chunked prefill: a later chunk of a long prompt onto a cache that already
// holds the earlier tokens packed.  Query row i of the chunk attends, in one
// softmax, the P0 cached keys as stored and the chunk's keys 0 .. i as given.
//
// Method: "RoPE-Aware Bit Allocation for KV-Cache Quantization" — the packed
// cache (review §1 "Packed-Cache") is what earlier chunks left; attention
// over it is the decode path's arithmetic.  Fusing the quantizer into an
// attention operator is named as future work on the LogQuant page (section
// "중요성 및 주장").
//
// The prefix is attended on the tensor cores in the codecs' own domains.
// For a key, q . k_hat = rho_k * sum_j q''_j c_j with c_j the centroid of
// codec coordinate j and q'' = BF(q[perm] * dewhiten * sign * 1/sqrt(piece))
// (BF: the per-piece butterflies, which are their own transpose); for the
// values, sum_t p_t v_hat_t = sign * BF(sum_t p_t rho_v,t c_t) / sqrt(128).
// A first kernel decodes each prefix token's packed records once into a
// workspace: its raw centroids (fp16-exact, codec order) for K and V and its
// two norms.  The attention kernel copies those rows by TMA like the chunk's
// own K/V, rotates its query rows once, scales the logits by the key norms in
// fp32 and the probabilities by the value norms, and takes the output row
// back to the value dims once, when the chunk's own tiles begin.  Query and
// probabilities are split into fp16 hi + lo parts (two MMAs each) so that the
// products keep about 22 bits, as in the decode path; each rotated query row
// is first scaled by a power of two to below 2^14, undone on its logits.
//
// Attention: one CTA takes 128 rows of one query head; 10 warps:
//   warps 0-3, 4-7  softmax warpgroups on the same rows (thread i = row i =
//              tensor-memory lane i), each taking 64 of a tile's 128 keys
//   warp 8     MMA issue (one thread), owner of the tensor memory
//   warp 9     TMA: Q, the prefix tiles and norms, the chunk's K/V tiles
// Tensor memory: S in two buffers (columns 0 and 128), O at 256, the rotated
// query's hi and lo parts at 384 and 448 (the A operand of the prefix S
// MMAs, so that only the key tile is read from shared memory; the chunk's
// own tiles take Q from shared memory); P overwrites the S it came from, 32
// keys per 32 columns: the hi parts of the chunk's 16 key pairs in its first
// 16 columns, the lo parts in the next 16.
// MMA order: S(0), S(1), then PV(j), S(j+2) for every tile j.
// Waits on O: a rescale at tile j waits for PV(j - 1) on the per-tile PV
// barrier (its parity names one phase there, S(j) having been issued after
// PV(j - 2)); the move to the value dims after the prefix and the final read
// wait on barriers committed once (PV of the last prefix tile; every MMA).
// The P barrier: the MMA thread waits for P(j) right after issuing S(j + 1),
// and the softmax can arrive P(j + 1) only once S(j + 1) has run and been
// read, so its phase is never two ahead of that wait (were it, the wait would
// run out and report the call as failed; no output would be wrong).
#include <cuda.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>

#include <cmath>
#include <mutex>
#include <type_traits>

#include "bgtq_internal.h"
#include "tc_common.cuh"

namespace bgtq {
namespace {

constexpr int kCkRows = 128;
constexpr int kCkKeys = 128;
constexpr int kCkThreads = 320;
constexpr uint32_t kCkTile = 128 * kD * 2;  // 32 KB
constexpr uint32_t kCkBox = kCkTile / 2;
constexpr uint32_t kCOffQ = 0;              // Q
constexpr uint32_t kCOffK = kCkTile;        // K stage s at + s kCkTile
constexpr uint32_t kCOffV = 3 * kCkTile;    // V stage s at + s kCkTile
constexpr uint32_t kCkSmem = 5 * kCkTile + 1024;
constexpr uint32_t kCColQ = 384;            // tensor-memory columns of the rotated query (hi; lo at + 64)
constexpr int kRawK = 4 * 3 + 1;            // words of a staged K record (bK <= 3) + a zero word
constexpr int kRawV = 8 * 4 + 1;            // words of a staged V pair record (bV <= 4) + a zero word
constexpr int kMmaWarp = 8, kTmaWarp = 9;
constexpr float kHeadroomC = 8.0f;
constexpr float kPvScale = 1.0f / 256.0f;   // prefix probabilities * rho_v are stored scaled by this

enum {
    kCQ = 0,        // Q copied
    kCQR = 1,       // rotated query written to tensor memory (128 arrivals)
    kCKF = 2,       // K tile of stage s copied, 2 + s
    kCVF = 4,       // V tile (and, for a prefix tile, its norms) of stage s copied
    kCKE = 6,       // K stage s free again (MMA commit)
    kCVE = 8,
    kCS = 10,       // S buffer b computed, 10 + b
    kCP = 12,       // P of the current tile written (256 arrivals)
    kCO = 13,       // PV of a tile done (one phase per tile; waited on only at a tile
                    // whose S wait proves PV of the tile before last done, so that the
                    // parity names one phase)
    kCDrain = 14,   // every MMA done (one phase)
    kCOPre = 15,    // PV of the last prefix tile done (one phase)
    kCNumBars = 16
};

struct CkParams {
    const __half* q;  // [B][H*G][C][128], the chunk's queries
    const __half* k;  // [B][H][C][128], the chunk's keys and values as given
    const __half* v;
    void* out;        // [B][H*G][C][128]
    int out_dtype;
    int C, H, G;
    float scale_log2;
    const int32_t* pos_start;  // [B]: prefix length P0 of each sequence
    int max_prefix;            // P0 bound of the workspace
    int pmax;                  // workspace rows per (sequence, head): max_prefix rounded up to 128
    // the decoded prefix (workspace): raw centroids [B][H][pmax][128] fp16, norms [B][H][pmax]
    __half* kh;
    __half* vh;
    float* rk;
    float* rv;
    // the packed cache
    const uint8_t* kc;
    const float* kn;
    const uint8_t* vc;
    const float* vn;
    CacheMap map;
    const HeadTab* heads;
    const float* cent;  // [9][256]
    int bk, bv;
    int32_t* status;
};

__device__ __forceinline__ uint32_t swz_off(int row, int col) {
    // element (row, col) of a [128][128] fp16 tile held as two 64-column boxes
    return (uint32_t)((col >> 6) * kCkBox + row * 128 + ((((col & 63) >> 3) ^ (row & 7)) << 4) + (col & 7) * 2);
}

// plain (untiled) bulk copy global -> shared completing on an mbarrier; both
// addresses 16-byte aligned, size a multiple of 16
__device__ __forceinline__ void bulk_copy(uint32_t dst, const void* src, uint32_t bytes, uint32_t bar) {
    asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(dst),
                 "l"(src), "r"(bytes), "r"(bar)
                 : "memory");
}

__device__ __forceinline__ void named_sync(int id, int n) { asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(n) : "memory"); }
// barrier over n threads that also ANDs a predicate across them
__device__ __forceinline__ bool named_sync_and(int id, int n, bool v) {
    uint32_t r;
    asm volatile(
        "{\n .reg .pred p, q;\n setp.ne.u32 p, %1, 0;\n bar.red.and.pred q, %2, %3, p;\n selp.u32 %0, 1, 0, q;\n}\n"
        : "=r"(r)
        : "r"((uint32_t)v), "r"(id), "r"(n)
        : "memory");
    return r != 0;
}

// Unnormalised butterflies over 128 values in registers; stage h acts on the
// pairs (j, j + h) with j < n[h] (the pieces larger than h form that prefix).
template <bool kAll>
__device__ __forceinline__ void butterflies128(float (&x)[kD], const int* nh) {
#pragma unroll
    for (int st = 0; st < 7; ++st) {
        const int h = 1 << st;
        const int lim = kAll ? kD : nh[st];
#pragma unroll
        for (int j = 0; j < kD; ++j) {
            if (j & h) continue;
            if (kAll || j < lim) {
                const float a = x[j], b = x[j + h];
                x[j] = a + b;
                x[j + h] = a - b;
            }
        }
    }
}


// Decode of the prefix into the workspace: thread r of block (tile, h, b)
// takes position 128 tile + r; positions from P0 up to the tile's end get
// zero rows and norms (the attention masks them; zeros keep its MMAs finite).
__global__ void __launch_bounds__(kCkKeys) chunk_prefix_decode_kernel(CkParams p) {
    __shared__ __half s_cent[(kWMax + 1) * 256];  // centroids, fp16-exact
    __shared__ uint32_t s_ktab[kD];               // K code j: bit position | width << 16
    __shared__ uint32_t s_rawk[kCkKeys][kRawK];   // staged K records
    __shared__ uint32_t s_rawv[kCkKeys / 2][kRawV];
    const int r = threadIdx.x, tile = blockIdx.x, h = blockIdx.y, b = blockIdx.z;
    const int P0 = p.pos_start[b];
    if (P0 < 0 || P0 > p.max_prefix || (int64_t)P0 + p.C > p.map.cap || tile * kCkKeys >= P0) return;
    const HeadTab* ht = p.heads + h;
    for (int i = r; i < (kWMax + 1) * 256; i += kCkKeys) s_cent[i] = __float2half_rn(p.cent[i]);
    {
        const int j = r;
        const int w = j < ht->n_coded ? ht->width[j] : 0;
        const int bit = w ? ht->pair_bit[j >> 1] + (j & 1) * w : 0;
        s_ktab[j] = (uint32_t)bit | ((uint32_t)w << 16);
    }
    const int rk = 4 * p.bk, rv = 8 * p.bv;
    const int pos = tile * kCkKeys + r;
    int64_t sl = -1;
    if (pos < P0) {
        sl = p.map.slot(b, h, pos);
        if (sl < 0 && p.status) atomicOr(p.status, BGTQ_STATUS_PAGE_RANGE);
    }
    // raw records into shared memory (the V pair record by the even key)
    if (sl >= 0) {
        const uint4* src = reinterpret_cast<const uint4*>(p.kc + sl * (16 * p.bk));
        for (int i = 0; i < p.bk; ++i) {
            const uint4 w4 = src[i];
            s_rawk[r][4 * i] = w4.x;
            s_rawk[r][4 * i + 1] = w4.y;
            s_rawk[r][4 * i + 2] = w4.z;
            s_rawk[r][4 * i + 3] = w4.w;
        }
    } else {
        for (int i = 0; i < rk; ++i) s_rawk[r][i] = 0u;
    }
    s_rawk[r][rk] = 0u;
    if ((r & 1) == 0) {
        if (sl >= 0) {
            const uint4* src = reinterpret_cast<const uint4*>(p.vc + (sl >> 1) * (32 * p.bv));
            for (int i = 0; i < 2 * p.bv; ++i) {
                const uint4 w4 = src[i];
                s_rawv[r >> 1][4 * i] = w4.x;
                s_rawv[r >> 1][4 * i + 1] = w4.y;
                s_rawv[r >> 1][4 * i + 2] = w4.z;
                s_rawv[r >> 1][4 * i + 3] = w4.w;
            }
        } else {
            for (int i = 0; i < rv; ++i) s_rawv[r >> 1][i] = 0u;
        }
        s_rawv[r >> 1][rv] = 0u;
    }
    __syncthreads();
    const size_t row = (((size_t)b * p.H + h) * p.pmax + pos);
    const bool live = sl >= 0;
    // K row: centroid of codec coordinate jj (codec order)
    uint4* kdst = reinterpret_cast<uint4*>(p.kh + row * kD);
#pragma unroll 1
    for (int c8 = 0; c8 < kD / 8; ++c8) {
        uint32_t packed[4];
#pragma unroll
        for (int e = 0; e < 4; ++e) {
            __half hv[2];
#pragma unroll
            for (int u = 0; u < 2; ++u) {
                const uint32_t t = s_ktab[8 * c8 + 2 * e + u];
                const uint32_t w = t >> 16, bit = t & 0xFFFFu;
                const uint32_t lo = s_rawk[r][bit >> 5], hi = s_rawk[r][(bit >> 5) + 1];
                const uint32_t code = __funnelshift_r(lo, hi, bit & 31u) & ((1u << w) - 1u);
                hv[u] = (w && live) ? s_cent[w * 256 + code] : __float2half_rn(0.0f);
            }
            packed[e] = (uint32_t)__half_as_ushort(hv[0]) | ((uint32_t)__half_as_ushort(hv[1]) << 16);
        }
        kdst[c8] = make_uint4(packed[0], packed[1], packed[2], packed[3]);
    }
    // V row: dim d holds code_even | code_odd << bV at bit 2 bV d
    uint4* vdst = reinterpret_cast<uint4*>(p.vh + row * kD);
    const uint32_t bvv = (uint32_t)p.bv, par_sh = (uint32_t)(r & 1) * bvv;
#pragma unroll 1
    for (int c8 = 0; c8 < kD / 8; ++c8) {
        uint32_t packed[4];
#pragma unroll
        for (int e = 0; e < 4; ++e) {
            __half hv[2];
#pragma unroll
            for (int u = 0; u < 2; ++u) {
                const uint32_t bit = 2u * bvv * (uint32_t)(8 * c8 + 2 * e + u) + par_sh;
                const uint32_t lo = s_rawv[r >> 1][bit >> 5], hi = s_rawv[r >> 1][(bit >> 5) + 1];
                const uint32_t code = __funnelshift_r(lo, hi, bit & 31u) & ((1u << bvv) - 1u);
                hv[u] = live ? s_cent[bvv * 256 + code] : __float2half_rn(0.0f);
            }
            packed[e] = (uint32_t)__half_as_ushort(hv[0]) | ((uint32_t)__half_as_ushort(hv[1]) << 16);
        }
        vdst[c8] = make_uint4(packed[0], packed[1], packed[2], packed[3]);
    }
    p.rk[row] = live ? p.kn[sl] : 0.0f;
    // the value norm times kPvScale (a power of two: exact), the factor the
    // attention gives each prefix probability
    p.rv[row] = live ? p.vn[sl] * kPvScale : 0.0f;
}

__global__ void __launch_bounds__(kCkThreads, 1)
    chunk_kernel(const __grid_constant__ CUtensorMap tq, const __grid_constant__ CUtensorMap tk,
                 const __grid_constant__ CUtensorMap tv, const __grid_constant__ CUtensorMap tkp,
                 const __grid_constant__ CUtensorMap tvp, CkParams p) {
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    __shared__ __align__(8) uint64_t s_bar[kCNumBars];
    __shared__ uint32_t s_tmem;
    __shared__ int s_abort;
    __shared__ uint8_t s_qperm[kD];               // rotated query: source dim of codec index j
    __shared__ float s_qscale[kD];                // dewhiten * sign * 1/sqrt(piece) (0 past n_coded)
    __shared__ float s_vsign[kD];
    __shared__ int s_nh[8];                       // butterfly stage h = 2^i: pairs j < s_nh[i]
    __shared__ __align__(16) float s_rho[2][2][kCkKeys];  // stage, (key, value) norms of the prefix keys
    __shared__ float s_mx[2][2][kCkRows];                 // row maxima of each warpgroup's half (tile parity)
    __shared__ float s_lsum[2][kCkRows];                  // row sums of each warpgroup's half
    __shared__ float s_qun[kCkRows];                      // the rotated query rows' power-of-two scaling

    const uint32_t sbase = (smem_u32(smem_raw) + 1023u) & ~1023u;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int hq = (int)blockIdx.x % (p.H * p.G);
    const int b = (int)blockIdx.x / (p.H * p.G);
    const int h = hq / p.G;
    const int nqb = (p.C + kCkRows - 1) / kCkRows;
    const int qb = nqb - 1 - (int)blockIdx.y;  // heaviest query blocks first
    const int q0 = qb * kCkRows;
    const int P0 = p.pos_start[b];
    const HeadTab* ht = p.heads + h;
    // a chunk past the capacity (the append flagged it and wrote nothing) or
    // a prefix past the workspace: zero rows
    if (P0 < 0 || (int64_t)P0 + p.C > p.map.cap || P0 > p.max_prefix) {
        if (P0 > p.max_prefix && tid == 0 && blockIdx.x == 0 && blockIdx.y == 0 && p.status)
            atomicOr(p.status, BGTQ_STATUS_SEQLEN_CAPACITY);
        if (tid < kCkRows && q0 + tid < p.C) {
            const size_t o = (((size_t)b * p.H * p.G + hq) * p.C + q0 + tid) * kD;
            for (int d = 0; d < kD; ++d) {
                if (p.out_dtype) static_cast<float*>(p.out)[o + d] = 0.0f;
                else static_cast<__half*>(p.out)[o + d] = __float2half_rn(0.0f);
            }
        }
        return;
    }
    const int np = (P0 + kCkKeys - 1) / kCkKeys;  // prefix tiles
    const int nc = qb + 1;                        // chunk tiles; the last holds the diagonal
    const int nt = np + nc;
    const uint32_t bar0 = smem_u32(&s_bar[0]);
    volatile int* abort_flag = &s_abort;
#define CBAR(i) (bar0 + 8u * (uint32_t)(i))

    // ---- set-up: barriers, tensor memory, the head's query-rotation tables
    if (tid == 0) {
        s_abort = 0;
        for (int i = 0; i < kCNumBars; ++i) mbar_init(CBAR(i), i == kCQR ? kCkRows : i == kCP ? 2 * kCkRows : 1);
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    if (warp == kMmaWarp) {
        asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(&s_tmem)),
                     "r"(512));
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;");
    }
    const int n_coded = ht->n_coded;
    for (int j = tid; j < kD; j += kCkThreads) {
        s_qperm[j] = ht->perm[j];
        s_qscale[j] = j < n_coded ? ht->dewhiten[j] * ht->sign_k[j] * ht->inv_sqrt[j] : 0.0f;
        s_vsign[j] = ht->sign_v[j];
    }
    if (warp == kTmaWarp) {
        for (int st = 0; st < 7; ++st) {
            int cnt = 0;
            for (int j = lane; j < kD; j += 32) cnt += (j < n_coded && (1 << ht->plog2[j]) > (1 << st)) ? 1 : 0;
            cnt = __reduce_add_sync(0xffffffffu, cnt);
            if (lane == 0) s_nh[st] = cnt;
        }
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = s_tmem;

    if (warp == kTmaWarp) {
        // ---- TMA: Q; prefix tiles (decoded rows and their norms); the
        // chunk's K/V tiles
        if (lane == 0) {
            const int qrow = (b * p.H * p.G + hq) * p.C + q0;
            const int krow = (b * p.H + h) * p.C;
            const int prow = (b * p.H + h) * p.pmax;
            mbar_expect_tx(CBAR(kCQ), kCkTile);
            for (int x = 0; x < 2; ++x) tma_load_2d(sbase + kCOffQ + x * kCkBox, &tq, 64 * x, qrow, CBAR(kCQ));
            int last_k[2] = {-1, -1}, last_v[2] = {-1, -1};
            int uses[2] = {0, 0};
            for (int j = 0; j < nt; ++j) {
                const int s = j & 1;
                const uint32_t par = (uint32_t)((j >> 1) - 1) & 1u;
                const bool pre = j < np;
                if (j >= 2 && !mbar_wait(CBAR(kCKE + s), par, abort_flag, p.status)) break;
                mbar_expect_tx(CBAR(kCKF + s), kCkTile);
                for (int x = 0; x < 2; ++x) {
                    if (pre)
                        tma_load_2d(sbase + kCOffK + s * kCkTile + x * kCkBox, &tkp, 64 * x, prow + j * kCkKeys, CBAR(kCKF + s));
                    else
                        tma_load_2d(sbase + kCOffK + s * kCkTile + x * kCkBox, &tk, 64 * x, krow + (j - np) * kCkKeys,
                                    CBAR(kCKF + s));
                }
                last_k[s] = uses[s];
                if (j >= 2 && !mbar_wait(CBAR(kCVE + s), par, abort_flag, p.status)) break;
                mbar_expect_tx(CBAR(kCVF + s), kCkTile + (pre ? 2u * kCkKeys * 4u : 0u));
                for (int x = 0; x < 2; ++x) {
                    if (pre)
                        tma_load_2d(sbase + kCOffV + s * kCkTile + x * kCkBox, &tvp, 64 * x, prow + j * kCkKeys, CBAR(kCVF + s));
                    else
                        tma_load_2d(sbase + kCOffV + s * kCkTile + x * kCkBox, &tv, 64 * x, krow + (j - np) * kCkKeys,
                                    CBAR(kCVF + s));
                }
                if (pre) {
                    bulk_copy(smem_u32(&s_rho[s][0][0]), p.rk + (size_t)prow + (size_t)j * kCkKeys, kCkKeys * 4, CBAR(kCVF + s));
                    bulk_copy(smem_u32(&s_rho[s][1][0]), p.rv + (size_t)prow + (size_t)j * kCkKeys, kCkKeys * 4, CBAR(kCVF + s));
                }
                last_v[s] = uses[s];
                ++uses[s];
            }
            // every copy issued has landed before the CTA ends
            mbar_wait(CBAR(kCQ), 0u, abort_flag, p.status, false);
            for (int s = 0; s < 2; ++s) {
                if (last_k[s] >= 0) mbar_wait(CBAR(kCKF + s), (uint32_t)last_k[s] & 1u, abort_flag, p.status, false);
                if (last_v[s] >= 0) mbar_wait(CBAR(kCVF + s), (uint32_t)last_v[s] & 1u, abort_flag, p.status, false);
            }
        }
        __syncwarp();
    } else if (warp == kMmaWarp) {
        // ---- MMA issue
        if (lane == 0) {
            constexpr uint32_t idS = instr_desc(kCkRows, kCkKeys, 0);
            constexpr uint32_t idO = instr_desc(kCkRows, kD, 1);
            int cnt_k[2] = {0, 0}, cnt_v[2] = {0, 0};
            bool ok = mbar_wait(CBAR(kCQ), 0, abort_flag, p.status);
            if (ok && np > 0) ok = mbar_wait(CBAR(kCQR), 0, abort_flag, p.status);
            auto issue_s = [&](int j) -> bool {
                const int s = j & 1;
                const uint32_t ka = sbase + kCOffK + s * kCkTile, d = tmem + 128u * (uint32_t)s;
                if (!mbar_wait(CBAR(kCKF + s), (uint32_t)(cnt_k[s]++) & 1u, abort_flag, p.status)) return false;
                tc_fence_after();
                if (j < np) {
                    // the rotated query's hi and lo parts from tensor memory
                    for (int part = 0; part < 2; ++part)
#pragma unroll
                        for (int k = 0; k < kD / 16; ++k) {
                            const uint32_t off = (uint32_t)(k >> 2) * kCkBox + (uint32_t)(k & 3) * 32;
                            mma_ts(d, tmem + kCColQ + 64u * (uint32_t)part + 8u * (uint32_t)k, smem_desc(ka + off, 16, 1024),
                                   idS, (part | k) ? 1u : 0u);
                        }
                } else {
#pragma unroll
                    for (int k = 0; k < kD / 16; ++k) {
                        const uint32_t off = (uint32_t)(k >> 2) * kCkBox + (uint32_t)(k & 3) * 32;
                        mma_ss(d, smem_desc(sbase + kCOffQ + off, 16, 1024), smem_desc(ka + off, 16, 1024), idS, k ? 1u : 0u);
                    }
                }
                mma_commit(CBAR(kCS + s));
                mma_commit(CBAR(kCKE + s));
                return true;
            };
            auto issue_pv = [&](int j) -> bool {
                const int s = j & 1;
                const uint32_t va = sbase + kCOffV + s * kCkTile, pa = tmem + 128u * (uint32_t)s;
                if (!mbar_wait(CBAR(kCP), (uint32_t)j & 1u, abort_flag, p.status)) return false;
                if (!mbar_wait(CBAR(kCVF + s), (uint32_t)(cnt_v[s]++) & 1u, abort_flag, p.status)) return false;
                tc_fence_after();
                const int parts = j < np ? 2 : 1;
                for (int part = 0; part < parts; ++part)
#pragma unroll
                    for (int k = 0; k < kCkKeys / 16; ++k)
                        mma_ts(tmem + 256u, pa + 32u * (k >> 1) + 8u * (k & 1) + 16u * part,
                               smem_desc(va + 2048u * k, kCkBox, 1024), idO, (j > 0 || part > 0 || k > 0) ? 1u : 0u);
                mma_commit(CBAR(kCO));
                mma_commit(CBAR(kCVE + s));
                if (j == np - 1) mma_commit(CBAR(kCOPre));
                return true;
            };
            if (ok) ok = issue_s(0);
            if (ok && nt > 1) ok = issue_s(1);
            for (int j = 0; ok && j < nt; ++j) {
                ok = issue_pv(j);
                if (ok && j + 2 < nt) ok = issue_s(j + 2);
            }
            mma_commit(CBAR(kCDrain));
            mbar_wait(CBAR(kCDrain), 0, abort_flag, p.status, false);
        }
        __syncwarp();
    } else {
        // ---- softmax: two warpgroups on the same rows; warpgroup hw takes
        // keys 64 hw .. 64 hw + 63 of every tile, thread r of each row q0 + r
        // of the chunk.  They exchange row maxima (and, at the end, row sums)
        // through shared memory and take every go/stop decision together at
        // named barrier 1 (an AND over both), so neither can be left waiting.
        const int hw = warp >> 2;
        const int r = tid & (kCkRows - 1);
        const int row = q0 + r;  // chunk-local
        const uint32_t lanes = (uint32_t)(32 * (warp & 3)) << 16;
        const float c = p.scale_log2;
        float q_unscale = 1.0f;  // prefix logits: times this power of two (the rotated query's scaling)
        bool ok = named_sync_and(1, 2 * kCkRows, mbar_wait(CBAR(kCQ), 0, abort_flag, p.status));
        if (ok && np > 0) {
            if (hw == 0) {
                // the rotated query q'' (codec order), split into fp16 hi + lo, over Q
                float x[kD];
                const uint8_t* qs = smem_raw + (sbase - smem_u32(smem_raw)) + kCOffQ;
    #pragma unroll
                for (int j = 0; j < kD; ++j) {
                    const float qv = __half2float(*reinterpret_cast<const __half*>(qs + swz_off(r, s_qperm[j] & (kD - 1))));
                    x[j] = qv * s_qscale[j];
                }
                int nh[7];
    #pragma unroll
                for (int st = 0; st < 7; ++st) nh[st] = s_nh[st];
                butterflies128<false>(x, nh);
                // the row scaled by a power of two to below 2^14 (the de-whitened
                // query can leave the fp16 range); the logits take it back exactly
                float amax = 0.0f;
    #pragma unroll
                for (int j = 0; j < kD; ++j) amax = fmaxf(amax, fabsf(x[j]));
                if (amax > 0.0f) {
                    int e2 = 0;
                    frexpf(amax, &e2);  // amax = f 2^e2, f in [0.5, 1)
                    const float up = ldexpf(1.0f, 14 - e2);
                    q_unscale = ldexpf(1.0f, e2 - 14);
    #pragma unroll
                    for (int j = 0; j < kD; ++j) x[j] *= up;
                }
                // into tensor memory, row r = lane r: column kCColQ + c holds
                // dims 2c, 2c + 1 of the hi part, kCColQ + 64 + c of the lo part
                const uint32_t tq_row = tmem + ((uint32_t)(32 * (warp & 3)) << 16) + kCColQ;
    #pragma unroll
                for (int c16 = 0; c16 < kD / 32; ++c16) {
                    uint32_t hp[16], lp[16];
    #pragma unroll
                    for (int e = 0; e < 16; ++e) {
                        const __half h0 = __float2half_rn(x[32 * c16 + 2 * e]), h1 = __float2half_rn(x[32 * c16 + 2 * e + 1]);
                        const __half l0 = __float2half_rn(x[32 * c16 + 2 * e] - __half2float(h0));
                        const __half l1 = __float2half_rn(x[32 * c16 + 2 * e + 1] - __half2float(h1));
                        hp[e] = (uint32_t)__half_as_ushort(h0) | ((uint32_t)__half_as_ushort(h1) << 16);
                        lp[e] = (uint32_t)__half_as_ushort(l0) | ((uint32_t)__half_as_ushort(l1) << 16);
                    }
                    tmem_st16(tq_row + 16u * (uint32_t)c16, hp);
                    tmem_st16(tq_row + 64u + 16u * (uint32_t)c16, lp);
                }
                tmem_wait_st();
                tc_fence_before();
                mbar_arrive(CBAR(kCQR));
                s_qun[r] = q_unscale;
            }
            named_sync(1, 2 * kCkRows);
            q_unscale = s_qun[r];
        }
        float m = 0.0f, l = 0.0f;  // l: this warpgroup's half of the row sum
        const uint32_t tO = tmem + lanes + 256u;
        // Tile j of the prefix (kPre) or of the chunk.  The combined decision
        // at its first named barrier is the only way out (false: both
        // warpgroups leave), so a warpgroup never leaves alone.
        auto tile = [&](int j, auto pre_tag) -> bool {
            constexpr bool kPre = decltype(pre_tag)::value;
            const int s = j & 1;
            const uint32_t tS = tmem + lanes + 128u * (uint32_t)s;
            // a prefix tile's norms arrive with its V tile
            const bool got = ok && mbar_wait(CBAR(kCS + s), (uint32_t)(j >> 1) & 1u, abort_flag, p.status) &&
                             (!kPre || mbar_wait(CBAR(kCVF + s), (uint32_t)(j >> 1) & 1u, abort_flag, p.status));
            if (!named_sync_and(1, 2 * kCkRows, got)) {
                ok = false;
                return false;
            }
            tc_fence_after();
            const int k0 = 64 * hw;  // the warpgroup's first key of the tile
            const int lim = (kPre ? P0 - 1 - j * kCkKeys                                    // keys past the prefix
                                  : (j == nt - 1 ? min(row, p.C - 1) - (j - np) * kCkKeys   // the chunk's diagonal
                                                 : kCkKeys)) - k0;
            // a prefix logit is S rho_k q_unscale: S rho_k here, q_unscale in
            // the tile's log2 scale (a positive factor: the maxima commute)
            const float cj = kPre ? c * q_unscale : c;
            float sv[64];
            float mxa[8];
            tmem_ld32(tS + k0, sv);
            tmem_wait_ld32(sv);
            tmem_ld32(tS + k0 + 32, sv + 32);
#pragma unroll
            for (int hh = 0; hh < 2; ++hh) {
                if (hh == 1) tmem_wait_ld32(sv + 32);
                if constexpr (kPre) {
                    const float4* rk4 = reinterpret_cast<const float4*>(&s_rho[s][0][k0 + 32 * hh]);
#pragma unroll
                    for (int k4 = 0; k4 < 8; ++k4) {
                        const float4 r4 = rk4[k4];
                        sv[32 * hh + 4 * k4] *= r4.x;
                        sv[32 * hh + 4 * k4 + 1] *= r4.y;
                        sv[32 * hh + 4 * k4 + 2] *= r4.z;
                        sv[32 * hh + 4 * k4 + 3] *= r4.w;
                    }
                }
                if (lim < 32 * hh + 31) {
#pragma unroll
                    for (int k = 32 * hh; k < 32 * hh + 32; ++k)
                        if (k > lim) sv[k] = -INFINITY;
                }
#pragma unroll
                for (int k = 32 * hh; k < 32 * hh + 32; ++k) mxa[k & 7] = k < 8 ? sv[k] : fmaxf(mxa[k & 7], sv[k]);
            }
            const float hmax = fmaxf(fmaxf(fmaxf(mxa[0], mxa[1]), fmaxf(mxa[2], mxa[3])),
                                     fmaxf(fmaxf(mxa[4], mxa[5]), fmaxf(mxa[6], mxa[7])));
            s_mx[s][hw][r] = hmax;
            named_sync(1, 2 * kCkRows);
            const float mt = fmaxf(hmax, s_mx[s][hw ^ 1][r]) * cj;
            float f = 1.0f;
            bool raise = false;
            if (j == 0) {
                m = mt;  // finite: key 0 (of the prefix, or of the chunk) is before every row
            } else if (mt > m + kHeadroomC) {
                f = ex2(m - mt);
                m = mt;
                l *= f;
                raise = true;
            }
            if (__any_sync(0xffffffffu, raise)) {
                // PV of tile j - 1 must be done before the warpgroup rescales its half
                // of O (S of this tile was issued after PV of tile j - 2, so kCO is at
                // phase j - 1 or past it and the parity names that phase)
                if (!__all_sync(0xffffffffu, mbar_wait(CBAR(kCO), (uint32_t)(j - 1) & 1u, abort_flag, p.status))) {
                    ok = false;  // both leave at the next tile's decision
                } else {
                    tc_fence_after();
#pragma unroll 1
                    for (int q4 = 2 * hw; q4 < 2 * hw + 2; ++q4) {
                        float o[32];
                        tmem_ld32(tO + 32 * q4, o);
                        tmem_wait_ld32(o);
                        uint32_t w[32];
#pragma unroll
                        for (int i = 0; i < 32; ++i) w[i] = __float_as_uint(o[i] * f);
                        tmem_st32(tO + 32 * q4, w);
                    }
                }
            }
            // P of each 32-key chunk of the half over that chunk's own 32
            // columns: hi parts in its first 16, lo parts (prefix tiles) in the next 16
            float ls[4] = {0.0f, 0.0f, 0.0f, 0.0f};
            const float4* rv4 = reinterpret_cast<const float4*>(&s_rho[s][1][k0]);
#pragma unroll
            for (int qh = 0; qh < 2; ++qh) {
                uint32_t hi[16], lo[16];
#pragma unroll
                for (int i2 = 0; i2 < 8; ++i2) {
                    const int k = 32 * qh + 4 * i2;
                    float pv[4];
#pragma unroll
                    for (int e = 0; e < 4; ++e) {
                        pv[e] = ex2(fmaf(sv[k + e], cj, -m));
                        ls[e] += pv[e];
                    }
                    if constexpr (kPre) {
                        // P' = p rho_v / 256 (the norms are stored scaled), split
                        // into fp16 hi + lo two at a time
                        const float4 r4 = rv4[k / 4];
                        const float a[4] = {pv[0] * r4.x, pv[1] * r4.y, pv[2] * r4.z, pv[3] * r4.w};
#pragma unroll
                        for (int e2 = 0; e2 < 2; ++e2) {
                            const __half2 h2 = __floats2half2_rn(a[2 * e2], a[2 * e2 + 1]);
                            const float2 hf = __half22float2(h2);
                            const __half2 l2 = __floats2half2_rn(a[2 * e2] - hf.x, a[2 * e2 + 1] - hf.y);
                            hi[2 * i2 + e2] = *reinterpret_cast<const uint32_t*>(&h2);
                            lo[2 * i2 + e2] = *reinterpret_cast<const uint32_t*>(&l2);
                        }
                    } else {
                        hi[2 * i2] = pack_h2(pv[0], pv[1]);
                        hi[2 * i2 + 1] = pack_h2(pv[2], pv[3]);
                    }
                }
                tmem_st16(tS + k0 + 32 * qh, hi);
                if constexpr (kPre) tmem_st16(tS + k0 + 32 * qh + 16, lo);
            }
            l += (ls[0] + ls[1]) + (ls[2] + ls[3]);
            tmem_wait_st();
            tc_fence_before();
            mbar_arrive(CBAR(kCP));
            return true;
        };
        for (int j = 0; j < np; ++j)
            if (!tile(j, std::true_type{})) break;
        if (np > 0) {  // (uniform; the chunk has at least one tile)
            // O leaves the value codec domain before the chunk's own tiles:
            // warpgroup 0 takes the whole row once PV of the last prefix tile
            // is done; both then pass one combined decision, so that neither
            // touches O before the transform is complete
            bool good = ok;
            if (hw == 0 && good) {
                good = __all_sync(0xffffffffu, mbar_wait(CBAR(kCOPre), 0u, abort_flag, p.status));
                if (good) {
                    tc_fence_after();
                    float o[kD];
#pragma unroll
                    for (int q4 = 0; q4 < kD / 32; ++q4) tmem_ld32(tO + 32 * q4, o + 32 * q4);
#pragma unroll
                    for (int q4 = 0; q4 < kD / 32; ++q4) tmem_wait_ld32(o + 32 * q4);
                    int nh_all[7];
                    butterflies128<true>(o, nh_all);
                    const float g = (1.0f / kPvScale) * 0.08838834764831845f;  // 1/sqrt(128)
#pragma unroll
                    for (int q4 = 0; q4 < kD / 32; ++q4) {
                        uint32_t w[32];
#pragma unroll
                        for (int i = 0; i < 32; ++i) w[i] = __float_as_uint(o[32 * q4 + i] * (g * s_vsign[32 * q4 + i]));
                        tmem_st32(tO + 32 * q4, w);
                    }
                    tmem_wait_st();
                    tc_fence_before();
                }
            }
            ok = named_sync_and(1, 2 * kCkRows, good);
            tc_fence_after();
        }
        if (ok)
            for (int j = np; j < nt; ++j)
                if (!tile(j, std::false_type{})) break;
        // the row sums of both halves; the output row, 64 columns per warpgroup
        s_lsum[hw][r] = l;
        // (the drain barrier has one phase: PV of the tile before last may
        // still run here, which a parity wait on kCO could not tell apart)
        const bool fin = ok && mbar_wait(CBAR(kCDrain), 0u, abort_flag, p.status);
        if (named_sync_and(1, 2 * kCkRows, fin)) {
            tc_fence_after();
            const float inv = 1.0f / (s_lsum[0][r] + s_lsum[1][r]);
            const size_t o0 = (((size_t)b * p.H * p.G + hq) * p.C + row) * kD;
#pragma unroll 1
            for (int q4 = 2 * hw; q4 < 2 * hw + 2; ++q4) {
                float o[32];
                tmem_ld32(tO + 32 * q4, o);
                tmem_wait_ld32(o);
                if (row >= p.C) continue;
                if (p.out_dtype) {
                    float4* dst = reinterpret_cast<float4*>(static_cast<float*>(p.out) + o0 + 32 * q4);
#pragma unroll
                    for (int i = 0; i < 8; ++i)
                        dst[i] = make_float4(o[4 * i] * inv, o[4 * i + 1] * inv, o[4 * i + 2] * inv, o[4 * i + 3] * inv);
                } else {
                    uint4* dst = reinterpret_cast<uint4*>(static_cast<__half*>(p.out) + o0 + 32 * q4);
#pragma unroll
                    for (int i = 0; i < 4; ++i)
                        dst[i] = make_uint4(pack_h2(o[8 * i] * inv, o[8 * i + 1] * inv),
                                            pack_h2(o[8 * i + 2] * inv, o[8 * i + 3] * inv),
                                            pack_h2(o[8 * i + 4] * inv, o[8 * i + 5] * inv),
                                            pack_h2(o[8 * i + 6] * inv, o[8 * i + 7] * inv));
                }
            }
        }
    }
#undef CBAR
    tc_fence_before();
    __syncthreads();
    if (warp == kMmaWarp) {
        tc_fence_after();
        asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(512));
    }
}

// The descriptors the kernel builds, checked field by field for every 1 KB
// aligned base it can have.
bool chunk_descriptors_valid() {
    if (!instr_desc_ok(instr_desc(kCkRows, kCkKeys, 0), 0) || !instr_desc_ok(instr_desc(kCkRows, kD, 1), 1)) return false;
    constexpr uint32_t kMaxSmem = 227u * 1024u;
    for (uint32_t base = 0; base + kCkSmem <= kMaxSmem + 1024; base += 1024)
        for (int k = 0; k < kD / 16; ++k) {
            const uint32_t off = (uint32_t)(k >> 2) * kCkBox + (uint32_t)(k & 3) * 32;
            for (uint32_t a : {base + kCOffQ + off, base + kCOffK + kCkTile + off})
                if (!smem_desc_ok(a, 16, 1024)) return false;
            if (!smem_desc_ok(base + kCOffV + kCkTile + (uint32_t)k * 2048, kCkBox, 1024)) return false;
        }
    return true;
}

int64_t chunk_pmax(int64_t max_prefix) { return (max_prefix + kCkKeys - 1) / kCkKeys * kCkKeys; }

}  // namespace

size_t prefill_chunk_workspace_bytes(const bgtq_plan& pl, int batch, int64_t max_prefix) {
    const size_t rows = (size_t)batch * pl.H * (size_t)chunk_pmax(max_prefix);
    return rows * (2 * kD * sizeof(__half) + 2 * sizeof(float));
}

cudaError_t launch_prefill_chunk(const bgtq_plan& pl, cudaStream_t s, const void* q, const void* k, const void* v,
                                 int batch, int c, const int32_t* pos_start, int64_t max_prefix, const bgtq_cache& cache,
                                 void* out, int out_dtype, float scale, void* ws, int32_t* status) {
    static std::mutex mu;
    static bool done[64] = {false};
    static const bool desc_ok = chunk_descriptors_valid();
    if (!desc_ok) return cudaErrorInvalidValue;
    const int64_t pmax = chunk_pmax(max_prefix);
    const uint64_t q_rows = (uint64_t)batch * pl.H * pl.G * (uint64_t)c;
    const uint64_t p_rows = (uint64_t)batch * pl.H * (uint64_t)pmax;
    const int nqb = (c + kCkRows - 1) / kCkRows;
    if (q_rows + kCkRows >= (1ull << 31) || p_rows + kCkKeys >= (1ull << 31) || nqb > 65535 ||
        (uint64_t)batch * pl.H * pl.G >= (1ull << 31) || pmax / kCkKeys > 0x7fffffff)
        return cudaErrorInvalidValue;
    int dev = 0;
    cudaGetDevice(&dev);
    if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
    {
        std::lock_guard<std::mutex> lock(mu);
        if (!done[dev]) {
            const cudaError_t e = cudaFuncSetAttribute(chunk_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kCkSmem);
            if (e != cudaSuccess) return e;
            done[dev] = true;
        }
    }
    CkParams p;
    p.q = static_cast<const __half*>(q);
    p.k = static_cast<const __half*>(k);
    p.v = static_cast<const __half*>(v);
    p.out = out;
    p.out_dtype = out_dtype;
    p.C = c;
    p.H = pl.H;
    p.G = pl.G;
    p.scale_log2 = scale * 1.4426950408889634f;
    p.pos_start = pos_start;
    p.max_prefix = (int)max_prefix;
    p.pmax = (int)pmax;
    char* w = static_cast<char*>(ws);
    p.kh = reinterpret_cast<__half*>(w);
    p.vh = reinterpret_cast<__half*>(w + p_rows * kD * sizeof(__half));
    p.rk = reinterpret_cast<float*>(w + 2 * p_rows * kD * sizeof(__half));
    p.rv = p.rk + p_rows;
    p.kc = static_cast<const uint8_t*>(cache.k_codes);
    p.kn = cache.k_norm;
    p.vc = static_cast<const uint8_t*>(cache.v_codes);
    p.vn = cache.v_norm;
    p.map = make_cache_map(cache, pl.H, batch, status);
    p.heads = pl.dev.heads;
    p.cent = pl.dev.cent;
    p.bk = pl.bk;
    p.bv = pl.bv;
    p.status = status;
    alignas(64) CUtensorMap tq, tk, tv, tkp, tvp;
    if (!rows_map(&tq, q, q_rows, kCkRows) || !rows_map(&tk, k, (uint64_t)batch * pl.H * c, kCkKeys) ||
        !rows_map(&tv, v, (uint64_t)batch * pl.H * c, kCkKeys))
        return cudaErrorInvalidValue;
    if (pmax > 0) {
        if (!rows_map(&tkp, p.kh, p_rows, kCkKeys) || !rows_map(&tvp, p.vh, p_rows, kCkKeys)) return cudaErrorInvalidValue;
        const dim3 dgrid((unsigned)(pmax / kCkKeys), (unsigned)pl.H, (unsigned)batch);
        chunk_prefix_decode_kernel<<<dgrid, kCkKeys, 0, s>>>(p);
        const cudaError_t e = cudaGetLastError();
        if (e != cudaSuccess) return e;
    } else {
        tkp = tk;  // no prefix tiles: never read
        tvp = tv;
    }
    const dim3 grid((unsigned)((uint64_t)batch * pl.H * pl.G), (unsigned)nqb, 1);
    chunk_kernel<<<grid, kCkThreads, kCkSmem, s>>>(tq, tk, tv, tkp, tvp, p);
    return cudaGetLastError();
}

}  // namespace bgtq
