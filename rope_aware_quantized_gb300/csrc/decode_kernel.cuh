// Split-K decode attention directly on the Block-GTQ packed cache, and the
// fused decode step (append the new token, then attend): the kernel template
// and its launch helpers, included by decode_attn.cu (contiguous caches) and
// decode_attn_paged.cu (paged caches).
//
// Method: "RoPE-Aware Bit Allocation for KV-Cache Quantization" — English
// abstract and review §1 "Packed-Cache" / Figure 2: attention is computed on
// the compressed K/V, no fp16 KV cache is materialised.
//
// Per CTA: one (sequence, KV head, token split), 4 warps; thread-block
// clusters of 8 consecutive splits.  Before waiting for the previous kernel
// (programmatic dependent launch) a CTA builds the lookup tables in shared
// memory (one copy per lane) and loads its per-lane lookup recipes.  After
// the wait: the fused step's owning CTA quantize-
// appends the new token; the G query heads are rotated once into the key
// codec domain (de-whitening, signs, blockwise Hadamard, 1/sqrt(piece),
// softmax scale and log2 e folded in), scaled per head by a power of two into
// the fp16 range, and split into fp16 hi + lo parts that form the 16 rows of
// the mma A operand (rows 0..7 hi, 8..15 lo).  Main loop, per warp and
// 16-token tile, tiles staged in shared memory by cp.async:
//   S^T = Q_hilo . K_hat^T     8 k-chunks x 2 token n-tiles of m16n8k16 mma;
//                              K_hat fragments come from a 64-bit window of
//                              the lane's K record slice: one shift + mask and
//                              one lookup in the lane's own copy of a pair
//                              table per 2 coords (codes of 4+ bits: one
//                              lookup per code in a single-code table)
//   logits = (hi + lo rows) * rho_K * scale, online softmax per head (exp2)
//   O^T += V_hat^T . P'        8 dim m-tiles of m16n8k16 mma, twice (P' =
//                              p*rho_V split hi + lo into two B operands);
//                              V_hat fragments come straight from the
//                              token-pair V records through the pair table
// Epilogue: each warp leaves its partial (m, l, acc) in shared memory; CTA
// rank r of the cluster reduces query head r over the cluster's 32 warp
// partials through distributed shared memory and writes one cluster partial
// to the workspace; the last cluster partial of each (sequence, head, query
// head) to arrive (atomic ticket) triggers the final log-sum-exp merge, the
// inverse value rotation and the output store.
#pragma once
#include <cooperative_groups.h>
#include <cuda_fp16.h>

#include <algorithm>
#include <cmath>
#include <map>
#include <mutex>

#include "bgtq_internal.h"
#include "encode.cuh"

namespace bgtq {

struct DecodeParams {
    const __half* q;
    uint8_t* kc;  // written only by the fused step (the new token)
    float* kn;
    uint8_t* vc;
    float* vn;
    int64_t cap;
    CacheMap map;  // record location of (sequence, head, position); paged or contiguous
    const int32_t* seq_lens;
    void* out;
    int out_dtype;
    float* part;
    uint32_t* count;
    const HeadTab* heads;
    const uint32_t* img_src;  // lookup tables: img_lane per-lane entries, then img_shared shared words
    int img_lane, img_shared;
    int img_ws;               // widest code the tables cover
    int img_bytes;            // bytes of the table region of the dynamic shared memory
    float scale_log2;
    float v_inv_sqrt;
    int H, G, n_split, tps;
    int slack;  // the newest token range is shorter by about this many tokens (multiple of 16)
    int32_t* status;
    // fused step: one new token per (sequence, KV head) quantize-appended at
    // pos_new[b] before attention (k_new == nullptr: attention only)
    const __half* k_new;
    const __half* v_new;
    const int32_t* pos_new;
    const float* thr;
    // fp16 recent-key ring [B][H][recent][128] (recent > 0): exact keys for
    // positions [seq - recent, seq); written by the fused step's append
    __half* k_recent;
    int64_t recent;
};

// Launches the paged-cache instances (defined in their own translation unit,
// so that the contiguous instances carry no paging code).
cudaError_t launch_decode_paged(const DecodeParams& p, dim3 grid, cudaStream_t s, int kind, int bk, int bv);

namespace {

namespace cg = cooperative_groups;

constexpr int kWarps = 4;
constexpr int kTile = 16;         // tokens per warp iteration; splits start on a tile boundary
constexpr int kCluster = 8;       // CTAs per thread-block cluster (consecutive splits of one head)
constexpr int kMaxClusters = 64;  // clusters per (sequence, head)
constexpr int64_t kMaxSplitTokens = 4096;  // longest token split of one CTA
constexpr int kWinPre = 256;               // longest fp16 key window of the precomputed-logit instance (1)
constexpr int kMaxTilesPerWarp = (int)(kMaxSplitTokens / (kWarps * 16));  // 16-token tiles of one warp
constexpr int kPartStride = 2 + kD;  // m, l, acc[128] per query head
// leading slots (width order 0, 8, 1, 9, ...) that may hold codes of width >= 4
// in the fast instances; the general instance treats every slot so
constexpr int kFastWide = 8;
// Softmax reference (log2 domain): set kLift above the largest logit when it
// is moved, moved again only when a logit passes it by more than kSlack.  The
// weights p then stay in (0, 2^kSlack] and the largest is >= 2^-kLift after a
// move, so P' = p * rho_V stays in the fp16 normal range for value norms
// from ~1e-3 to ~4e3, and the accumulator is rescaled only when the maximum
// grows by more than kLift + kSlack.
constexpr float kLift = 4.0f;
constexpr float kSlack = 4.0f;


// (not volatile: a pure register operation the compiler may schedule freely)
__device__ __forceinline__ void mma16816(float (&c)[4], const uint32_t (&a)[4], uint32_t b0, uint32_t b1) {
    asm(
        "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, {%0,%1,%2,%3};\n"
        : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
        : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

// Programmatic dependent launch: let the next kernel in the stream start its
// own set-up now / wait until the previous kernel's results are visible.
__device__ __forceinline__ void pdl_trigger() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }

// Ticket of the split merge: fetch-and-add with release (the CTA's partial,
// ordered before it by a CTA barrier, is visible before the count moves) and
// acquire (the last arriver then sees every other partial) at GPU scope.
__device__ __forceinline__ unsigned ticket_acq_rel(unsigned* ptr) {
    unsigned old;
    asm volatile("atom.add.acq_rel.gpu.u32 %0, [%1], 1;" : "=r"(old) : "l"(ptr) : "memory");
    return old;
}

__device__ __forceinline__ uint32_t h2_bits(__half2 h) { return *reinterpret_cast<uint32_t*>(&h); }

// hi = fp16(x), lo = fp16(x - hi) for a pair of values
__device__ __forceinline__ void split_hilo(float x0, float x1, uint32_t& hi, uint32_t& lo) {
    const __half2 h = __floats2half2_rn(x0, x1);
    const float2 hf = __half22float2(h);
    hi = h2_bits(h);
    lo = h2_bits(__floats2half2_rn(x0 - hf.x, x1 - hf.y));
}

__device__ __forceinline__ uint32_t lds32(const uint32_t* tab, uint32_t byte) {
    return *reinterpret_cast<const uint32_t*>(reinterpret_cast<const char*>(tab) + byte);
}

__device__ __forceinline__ float fast_exp2(float x) {
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

// 64-bit windows of one token's K lane slice (BK words): slots 0..7 read the
// slice shifted left by 7 bits, slots 8..15 its upper words (see KSlot).
template <int BK>
__device__ __forceinline__ uint64_t kwin_lo(const uint32_t (&kw)[BK]) {
    if constexpr (BK >= 2) return ((((uint64_t)kw[1]) << 32) | kw[0]) << 7;
    else return ((uint64_t)kw[0]) << 7;
}
template <int BK>
__device__ __forceinline__ uint64_t kwin_hi(const uint32_t (&kw)[BK]) {
    if constexpr (BK == 3) return (((uint64_t)kw[2]) << 32) | kw[1];
    else if constexpr (BK == 2) return (((uint64_t)kw[1]) << 32) | kw[0];
    else return (uint64_t)kw[0];
}

// Decoded fp16 pair of one K slot: one lookup in the lane's copy of a pair
// table or, for slots whose codes may be 4 bits or wider (kMayWide), a second
// lookup of the second code in the single table.  A pair-table slot has
// wsh = 0: its second lookup repeats the first and the byte permutation
// keeps that word whole; a single-table entry holds its value in both halves,
// so the permutation joins the first code's low half to the second's high.
template <bool kMayWide>
__device__ __forceinline__ uint32_t k_lookup(uint64_t win, uint32_t sh, uint32_t mask, uint32_t base, uint32_t wsh,
                                             const uint32_t* s_tab) {
    const uint32_t x = (uint32_t)(win >> sh);
    const uint32_t v0 = lds32(s_tab, (x & mask) | base);
    if constexpr (!kMayWide) return v0;
    const uint32_t v1 = lds32(s_tab, ((x >> wsh) & mask) | base);
    return __byte_perm(v0, v1, 0x7610);
}

// Rank of slot S in the lane's width order (slots 0, 8, 1, 9, ...).
template <int S>
__host__ __device__ constexpr int slot_rank() { return S < 8 ? 2 * S : 2 * (S - 8) + 1; }

// Decoded fp16 pair (even token, odd token) of V codec dim 16 g + J from the
// lane group's BV words of a token-pair record (compile-time bit position):
// the field is brought to bit 7 and looked up in the lane's pair table
// (BV <= 3), or its two codes in the width-4 single table (BV = 4).
template <int BV, int J>
__device__ __forceinline__ uint32_t v_field(const uint32_t (&vw)[BV], uint32_t vbase, const uint32_t* s_tab) {
    constexpr int FB = 2 * BV;
    constexpr int O = FB * J;
    constexpr int WI = O >> 5, SH = O & 31;
    uint32_t x;
    if constexpr (SH + FB <= 32) {
        if constexpr (SH >= 7)
            x = vw[WI] >> (SH - 7);
        else
            x = vw[WI] << (7 - SH);
    } else {
        x = __funnelshift_r(vw[WI], vw[WI + 1 < BV ? WI + 1 : WI], SH - 7);
    }
    if constexpr (BV <= kPairTableMaxW) {
        constexpr uint32_t MASK = ((1u << FB) - 1u) << 7;
        return lds32(s_tab, (x & MASK) | vbase);
    } else {
        constexpr uint32_t MASK = ((1u << BV) - 1u) << 7;
        const uint32_t v0 = lds32(s_tab, (x & MASK) | vbase);
        const uint32_t v1 = lds32(s_tab, ((x >> BV) & MASK) | vbase);
        return __byte_perm(v0, v1, 0x7610);
    }
}

// S^T += Q_hilo . K_hat^T for k-chunk C (slots 2C, 2C+1) of both 8-token
// groups of the tile.
template <int NW, int C>
__device__ __forceinline__ void s_chunk(float (&sacc)[2][4], const uint32_t (&qa)[8][4], const uint64_t (&wl)[2],
                                        const uint64_t (&wh)[2], const uint32_t (&ksh)[16], const uint32_t (&kmask)[16],
                                        const uint32_t (&kbase)[16], const uint32_t (&kwsh)[16], const uint32_t* s_tab) {
    constexpr int S0 = 2 * C, S1 = 2 * C + 1;
    constexpr bool W0 = slot_rank<S0>() < NW, W1 = slot_rank<S1>() < NW;
#pragma unroll
    for (int nt = 0; nt < 2; ++nt) {
        const uint64_t win = C < 4 ? wl[nt] : wh[nt];
        const uint32_t b0 = k_lookup<W0>(win, ksh[S0], kmask[S0], kbase[S0], kwsh[S0], s_tab);
        const uint32_t b1 = k_lookup<W1>(win, ksh[S1], kmask[S1], kbase[S1], kwsh[S1], s_tab);
        mma16816(sacc[nt], qa[C], b0, b1);
    }
}

// O^T += V_hat^T . P' for dim tile MT (codec dims 16 g + 2 MT and + 1 of the
// lane groups g = 0..7): A = the decoded value pairs of token pairs t and
// t + 4, B = the weights P' of the 16 tokens split hi + lo (two mma).
template <int BV, int MT>
__device__ __forceinline__ void pv_mtile(float (&acc)[8][4], const uint32_t (&pb)[2][2], const uint32_t (&vw)[2][BV],
                                         uint32_t vbase, const uint32_t* s_tab) {
    const uint32_t a[4] = {v_field<BV, 2 * MT>(vw[0], vbase, s_tab), v_field<BV, 2 * MT + 1>(vw[0], vbase, s_tab),
                           v_field<BV, 2 * MT>(vw[1], vbase, s_tab), v_field<BV, 2 * MT + 1>(vw[1], vbase, s_tab)};
    mma16816(acc[MT], a, pb[0][0], pb[0][1]);
    mma16816(acc[MT], a, pb[1][0], pb[1][1]);
}

// Blockwise Hadamard butterflies over the warp's 128 slots (lane L holds
// slots 4L..4L+3): stage h pairs (j, j+h) inside pieces larger than h.
__device__ __forceinline__ void rotate_warp(float (&x)[4], const int (&plog2)[4], int lane) {
#pragma unroll
    for (int h = 1; h <= 2; h <<= 1) {
        float y[4];
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const float o = x[i ^ h];
            y[i] = (1 << plog2[i]) > h ? ((i & h) ? o - x[i] : x[i] + o) : x[i];
        }
#pragma unroll
        for (int i = 0; i < 4; ++i) x[i] = y[i];
    }
#pragma unroll
    for (int h = 4; h < kD; h <<= 1) {
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const float o = __shfl_xor_sync(0xffffffffu, x[i], h >> 2);
            if ((1 << plog2[i]) > h) x[i] = ((4 * lane + i) & h) ? o - x[i] : x[i] + o;
        }
    }
}

// Staging of 16-token tiles in shared memory: every warp keeps kStages
// tiles in flight with cp.async (enough bytes in flight per SM to cover the
// HBM latency), then reads its operands from the staged copy.  One staged
// tile: 16 K records, 8 V pair records, 16 key norms, 16 value norms.
constexpr int kStages = 4;

template <int BK, int BV>
struct StageLayout {
    static constexpr int kK = 16 * 16 * BK;
    static constexpr int kV = 8 * 32 * BV;
    static constexpr int kN = kK + kV;  // key norms, then value norms
    static constexpr int kBytes = kN + 2 * 16 * 4;
    static_assert(kK % 16 == 0 && kV % 16 == 0, "16-byte copies");
};

// Dynamic shared memory of decode_kernel<BK, BV>: the lookup tables (img_bytes
// of them, at least the size of the per-warp and per-CTA partials that
// reuse the region after the main loop), the rotated queries, then kStages
// staged tiles per warp (whose region also holds the tables' compact source
// during the set-up).
constexpr int kPartBytes = (kWarps + 1) * 8 * kPartStride * 4;
constexpr int kQBytes = 8 * kD * 4;  // rotated queries
inline int decode_table_bytes(int ws) {
    const int b = (image_bytes(ws) + 127) / 128 * 128;
    return b > kPartBytes ? b : (kPartBytes + 127) / 128 * 128;
}
template <int BK, int BV>
constexpr int decode_stage_bytes() {
    return kWarps * kStages * StageLayout<BK, BV>::kBytes;
}
template <int BK, int BV>
int decode_smem_bytes(int ws) {
    return decode_table_bytes(ws) + kQBytes + decode_stage_bytes<BK, BV>();
}
static_assert(kWarps * kStages * StageLayout<1, 1>::kBytes >= kImageMaxWords * 4, "the table source fits the staging region");

// 16-byte (or, for the norms, 4-byte) asynchronous copy global -> shared;
// `valid` false copies nothing and zero-fills.
__device__ __forceinline__ void cp_async16(uint32_t dst, const void* src, bool valid) {
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;\n" ::"r"(dst), "l"(src), "r"(valid ? 16 : 0)
                 : "memory");
}
__device__ __forceinline__ void cp_async4(uint32_t dst, const void* src, bool valid) {
    asm volatile("cp.async.ca.shared.global [%0], [%1], 4, %2;\n" ::"r"(dst), "l"(src), "r"(valid ? 4 : 0) : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;\n" ::: "memory"); }
template <int N>
__device__ __forceinline__ void cp_async_wait() { asm volatile("cp.async.wait_group %0;\n" ::"n"(N) : "memory"); }

// The warp copies tile [T0, T0 + 16) into the stage at shared address `st`;
// tokens at or beyond `seq` are zero-filled (never read from global).  The
// tile's records start at token slot `tb` of kc/vc/kn/vn (a tile never
// straddles a page).
template <int BK, int BV>
__device__ __forceinline__ void stage_tile(uint32_t st, const uint8_t* kc, const uint8_t* vc, const float* kn,
                                           const float* vn, int64_t tb, int T0, int seq, int lane) {
    using SL = StageLayout<BK, BV>;
    const uint8_t* ksrc = kc + tb * (16 * BK);
#pragma unroll
    for (int c = lane; c < 16 * BK; c += 32) {
        const bool ok = T0 + c / BK < seq;
        cp_async16(st + 16 * c, ok ? ksrc + 16 * c : kc, ok);
    }
    const uint8_t* vsrc = vc + (tb >> 1) * (32 * BV);
#pragma unroll
    for (int c = lane; c < 16 * BV; c += 32) {
        const bool ok = T0 + 2 * (c / (2 * BV)) < seq;
        cp_async16(st + SL::kK + 16 * c, ok ? vsrc + 16 * c : vc, ok);
    }
    const bool ok = T0 + (lane & 15) < seq;
    const float* nsrc = lane < 16 ? kn : vn;
    cp_async4(st + SL::kN + 4 * lane, ok ? nsrc + tb + (lane & 15) : nsrc, ok);
}

// Operands of one 16-token tile for one lane, read from its staged copy.
template <int BK, int BV>
struct TileRegs {
    uint32_t kw[2][BK];  // K record slice words of tokens T0 + g and T0 + 8 + g
    float rk[2][2];      // key norms of tokens T0 + 8 nt + 2 t + e
    float rv[2][2];      // value norms of the same tokens
    uint32_t vw[2][BV];  // lane-group words of V pair records T0/2 + t and T0/2 + 4 + t

    __device__ __forceinline__ void read(const uint8_t* st, int g, int t) {
        using SL = StageLayout<BK, BV>;
#pragma unroll
        for (int nt = 0; nt < 2; ++nt) {
            const uint32_t* src = reinterpret_cast<const uint32_t*>(st + (8 * nt + g) * (16 * BK)) + BK * t;
#pragma unroll
            for (int i = 0; i < BK; ++i) kw[nt][i] = src[i];
            const float2 k2 = *reinterpret_cast<const float2*>(st + SL::kN + 4 * (8 * nt + 2 * t));
            const float2 v2 = *reinterpret_cast<const float2*>(st + SL::kN + 64 + 4 * (8 * nt + 2 * t));
            rk[nt][0] = k2.x;
            rk[nt][1] = k2.y;
            rv[nt][0] = v2.x;
            rv[nt][1] = v2.y;
        }
#pragma unroll
        for (int r = 0; r < 2; ++r) {
            const uint32_t* src = reinterpret_cast<const uint32_t*>(st + SL::kK + (4 * r + t) * (32 * BV)) + BV * g;
#pragma unroll
            for (int i = 0; i < BV; ++i) vw[r][i] = src[i];
        }
    }
};

// Fused step: quantize-append the new token of (sequence, KV head) `unit` at
// `pos`, warp 0 the key and warp 1 the value (the same encoder steps as the
// quantize-append kernel, so the codes are identical).  The value record of
// the token pair is merged in place with atomic AND/OR.
template <int BK, int BV>
__device__ __forceinline__ void append_new_token(const DecodeParams& p, const EncLane& el, size_t unit, int64_t sl, int pos,
                                                 const float* s_thr, uint32_t (*s_enc)[8 * kPairMaxW], int warp,
                                                 int lane) {
    if (warp == 0) {
        const __half* row = p.k_new + unit * kD;
        if (p.recent > 0)  // fp16 recent-key ring: the new key as given, slot pos mod W
            *(reinterpret_cast<uint2*>(p.k_recent + (unit * p.recent + pos % p.recent) * kD) + lane) =
                *(reinterpret_cast<const uint2*>(row) + lane);
        float x[1][4];
#pragma unroll
        for (int k = 0; k < 4; ++k) x[0][k] = __fmul_rn(__half2float(row[el.src[k]]), el.wh[k]);
        for (int k = lane; k < 8 * kPairMaxW; k += 32) s_enc[0][k] = 0;
        __syncwarp();
        int code[1][4];
        float rho[1];
        warp_encode_n<1>(x, el.sg, el.pl, el.is, el.wd, el.n_coded, s_thr, code, rho);
        pack_k_fields(s_enc[0], code[0], el, lane);
        __syncwarp();
        uint32_t* dst = reinterpret_cast<uint32_t*>(p.kc + sl * (16 * BK));
        if (lane < 4 * BK) dst[lane] = s_enc[0][lane];
        if (lane == 0) p.kn[sl] = rho[0];
    } else if (warp == 1) {
        const uint2 raw = *(reinterpret_cast<const uint2*>(p.v_new + unit * kD) + lane);
        const float2 a = __half22float2(*reinterpret_cast<const __half2*>(&raw.x));
        const float2 c = __half22float2(*reinterpret_cast<const __half2*>(&raw.y));
        float x[1][4] = {{a.x, a.y, c.x, c.y}};
        for (int k = lane; k < 8 * kPairMaxW; k += 32) {
            s_enc[1][k] = 0;
            s_enc[2][k] = 0;
        }
        __syncwarp();
        int code[1][4];
        float rho[1];
        warp_encode_n<1>(x, el.sg, el.pl, el.is, el.wd, kD, s_thr, code, rho);
        pack_v_fields(s_enc[1], s_enc[2], code[0], pos & 1, BV, lane);
        __syncwarp();
        uint32_t* vdst = reinterpret_cast<uint32_t*>(p.vc + (sl >> 1) * (32 * BV));
        for (int k = lane; k < 8 * BV; k += 32) {
            atomicAnd(vdst + k, ~s_enc[2][k]);
            atomicOr(vdst + k, s_enc[1][k]);
        }
        if (lane == 0) p.vn[sl] = rho[0];
    }
}

// Token slot of the new token of a fused step; an out-of-range page index
// is flagged and the append skipped.
__device__ __forceinline__ int64_t new_token_slot(const DecodeParams& p, int b, int h, int pos) {
    const int64_t sl = p.map.slot(b, h, pos);
    if (sl < 0 && p.status) atomicOr(p.status, BGTQ_STATUS_PAGE_RANGE);
    return sl;
}

__device__ __forceinline__ void cluster_arrive() { asm volatile("barrier.cluster.arrive.release.aligned;" ::: "memory"); }
__device__ __forceinline__ void cluster_wait() { asm volatile("barrier.cluster.wait.acquire.aligned;" ::: "memory"); }

template <bool B>
struct BoolTag {
    static constexpr bool value = B;
};

// Instances (kKind): 0 = fast (slots 0 and 8 alone may hold codes wider
// than the pair tables; no recent-key buffer), 1 = fast with an fp16
// recent-key buffer of at most kWinPre keys (their exact logits computed
// ahead of the main loop), 2 = general (any slot wide, any buffer); kPaged:
// the cache is paged.  The buffer and paging paths are separate instances
// so that the instances without them carry none of their code.
template <int BK, int BV, int kKind, bool kPaged>
__global__ void __launch_bounds__(kWarps * 32, 2) decode_kernel(DecodeParams p) {
    constexpr int NW = kKind == 2 ? 16 : kFastWide;  // leading slots that may hold codes of width >= 4
    constexpr bool kWinPath = kKind >= 1;  // fp16 recent-key buffer supported
    constexpr bool kWinPre1 = kKind == 1;  // its logits computed ahead (window <= kWinPre)
    constexpr bool kWinLoop = kKind == 2;  // its tiles in a second loop
    extern __shared__ __align__(16) uint8_t dsmem[];
    uint32_t* s_tab = reinterpret_cast<uint32_t*>(dsmem);
    float (*s_q)[kD] = reinterpret_cast<float (*)[kD]>(dsmem + p.img_bytes);
    uint8_t* s_stage = dsmem + p.img_bytes + kQBytes;
    __shared__ float s_qunscale[8];
    __shared__ int s_last;
    __shared__ float s_thr[kThrCompact];                 // fused step: encoder thresholds
    __shared__ uint32_t s_enc[3][8 * kPairMaxW];          // fused step: records being assembled
    __shared__ uint2 s_qo[8][32];                         // recent-key buffer: A fragments of q as given
    __shared__ float s_wlog[kWinPre1 ? 8 : 1][kWinPre1 ? kWinPre : 1];  // instance 1: exact window logits (log2 domain)
    __shared__ int64_t s_pslot[kPaged ? kWarps : 1][kPaged ? kMaxTilesPerWarp : 1];  // paged: tile slots
    // after the main loop the table region holds the per-warp partials of
    // the 8 query heads (m, l, acc[128]) that the cluster reads
    // and then the CTA's merged partial of the 8 heads
    float (*s_wp)[8][kPartStride] = reinterpret_cast<float (*)[8][kPartStride]>(s_tab);
    float (*s_cp)[kPartStride] = reinterpret_cast<float (*)[kPartStride]>(s_tab + kWarps * 8 * kPartStride);

    // The next kernel may launch right away; everything this kernel reads
    // that an earlier kernel may still be writing (q, the cache, the
    // workspace) is read only after pdl_wait().  seq_lens is never written by
    // this library's kernels.  Every CTA passes pdl_wait() before it exits.
    pdl_trigger();
    const int split = blockIdx.x, h = blockIdx.y, b = blockIdx.z;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31, g = lane >> 2, t = lane & 3;
    const int G = p.G;
    const size_t unit = (size_t)b * p.H + h;
    int seq = p.seq_lens[b];
    if (seq < 0 || (int64_t)seq > p.cap) {
        pdl_wait();
        if (tid == 0 && split == 0 && h == 0 && p.status) {
            atomicOr(p.status, BGTQ_STATUS_SEQLEN_CAPACITY);
            debug_in_range(false, p.status);  // records past the capacity
        }
        seq = seq < 0 ? 0 : (int)p.cap;
    }
    // Token ranges, newest first: split 0 attends [a0, seq) with a0 the
    // multiple of 16 at or above seq - (tps - slack), split s >= 1 the tps
    // tokens [a0 - s tps, a0 - (s - 1) tps) (the oldest one clipped at 0).
    // CTAs start in split order, so the newest tokens, and in a fused step
    // the append, go to the CTA that starts first, and its range is shorter
    // by about `slack` tokens to make up for the append.
    const int a0 = max(0, (seq - p.tps + p.slack + 15) & ~15);
    const int n_active = 1 + (a0 + p.tps - 1) / p.tps;
    const int n_clusters = (n_active + kCluster - 1) / kCluster;
    const int cid = split / kCluster;
    // Fused step: the CTA whose token range holds the new position appends
    // the new token before attending (split 0 when the position is not
    // attended).  pos_new is read before the wait, like seq_lens.
    bool owner = false, pos_bad = false;
    int pos = 0;
    EncLane el;
    if (p.k_new) {
        pos = p.pos_new[b];
        pos_bad = pos < 0 || (int64_t)pos + 1 > p.cap;
        owner = !pos_bad && split == (pos < seq && pos < a0 ? 1 + (a0 - 1 - pos) / p.tps : 0);
        if (owner) {
            stage_thresholds(s_thr, p.thr, tid, kWarps * 32);
            if (warp < 2) enc_lane_load(el, p.heads + h, warp == 0, BV, p.v_inv_sqrt, lane);
            __syncthreads();
        }
    }
    if (seq == 0) {
        pdl_wait();
        if (pos_bad && split == 0 && h == 0 && tid == 0 && p.status) {
            atomicOr(p.status, BGTQ_STATUS_APPEND_CAPACITY);
            debug_in_range(false, p.status);  // a new position past the capacity
        }
        if (owner) {
            const int64_t sl = new_token_slot(p, b, h, pos);
            if (sl >= 0) append_new_token<BK, BV>(p, el, unit, sl, pos, s_thr, s_enc, warp, lane);
        }
        if (split == 0) {
            for (int i = tid; i < G * kD; i += kWarps * 32) {
                const size_t o = ((size_t)b * p.H * G + (size_t)h * G) * kD + i;
                if (p.out_dtype) static_cast<float*>(p.out)[o] = 0.0f;
                else static_cast<__half*>(p.out)[o] = __float2half_rn(0.0f);
            }
        }
        return;  // every CTA of this (sequence, head) leaves here
    }
    if (cid >= n_clusters) {  // the whole cluster is past the sequence
        pdl_wait();
        return;
    }
    cg::cluster_group cluster = cg::this_cluster();
    const int crank = (int)cluster.block_rank();
    const bool active = split < n_active;
    const HeadTab* ht = p.heads + h;
    const int t_begin = !active ? seq : split == 0 ? a0 : max(0, a0 - split * p.tps);
    const int t_end = !active ? seq : split == 0 ? seq : a0 - (split - 1) * p.tps;
    const int wstart = p.recent > 0 ? max(0, seq - (int)p.recent) : seq;  // first position of the fp16 keys
    const int wlo = max(t_begin, wstart);  // the range's first window token (instance 1: s_wlog column 0)
    // record bases: the (sequence, head) row of a contiguous cache (token
    // slot = position), the pools of a paged one (token slot per tile)
    constexpr bool paged = kPaged;
    const size_t ubase = paged ? 0 : unit * (size_t)p.cap;
    const uint8_t* kc = p.kc + ubase * (16 * BK);
    const uint8_t* vc = p.vc + (ubase / 2) * (32 * BV);
    const float* kn = p.kn + ubase;
    const float* vn = p.vn + ubase;
    // token slot of the tile at position T0 (16-token tiles never straddle a
    // page; an out-of-range page index is flagged and page 0 read instead)
    // (no branch on the page index: the prologue flags bad ones, so the
    // page-table load can be issued a tile ahead of its use)
    auto tile_slot = [&](int T0) -> int64_t {
        if constexpr (!kPaged) return T0;
        const int64_t sl = p.map.slot(b, h, T0);
        return sl >= 0 ? sl : ((int64_t)h << p.map.lp) + (T0 & ((1 << p.map.lp) - 1));
    };
    // warp w takes tiles T0 = t_begin + 16 w + kStep k; kStages - 1 of them are
    // being copied while one is processed
    constexpr int kStep = kWarps * kTile;
    const int T0w = t_begin + warp * kTile;
    int n_tiles = active && T0w < t_end ? (t_end - T0w + kStep - 1) / kStep : 0;
    if (kPaged && n_tiles > kMaxTilesPerWarp) {  // excluded by the host's capacity check
        if (lane == 0 && p.status) atomicOr(p.status, BGTQ_STATUS_SEQLEN_CAPACITY);
        n_tiles = kMaxTilesPerWarp;
    }
    // paged: the token slots of all the warp's tiles (at most kMaxTilesPerWarp:
    // a paged cache holds at most kMaxSplitTokens * kCluster * kMaxClusters
    // positions, so a split is at most kMaxSplitTokens long) and of the new
    // token, looked up before the wait (the page table is read like seq_lens),
    // so that the main loop only reads a slot from shared memory
    int64_t sl_new = 0;
    if constexpr (kPaged) {
        for (int k = lane; k < n_tiles && k < kMaxTilesPerWarp; k += 32) s_pslot[warp][k] = tile_slot(T0w + k * kStep);
        __syncwarp();
        if (owner) sl_new = p.map.slot(b, h, pos);
    }

    // ---- plan-static set-up, before waiting for the previous kernel: the
    // lookup tables, the per-lane recipes
    const int n_coded = ht->n_coded;
    int q_pl[4], q_src[4];
    float q_f[4], q_sc[4];
    uint32_t ksh[16], kmask[16], kbase[16], kwsh[16];
    uint32_t slot_pairs[4];
    // (no L2 prefetch of the token range before the wait: under programmatic
    // dependent launch it competes with the previous kernel's own reads)
    if (kPaged && active) {
        // paged: thread i checks the page-table entry of page i of the range
        // (the page table is read before the wait, like seq_lens); the main
        // loop reads page 0 in place of a bad one
        const int lp = p.map.lp;
        const int pg0 = t_begin >> lp, pg1 = (t_end - 1) >> lp;
        for (int pi = pg0 + tid; pi <= pg1; pi += kWarps * 32) {
            const int a = (int)max((int64_t)t_begin, (int64_t)pi << lp);
            if (p.map.slot(b, h, a) < 0 && p.status) atomicOr(p.status, BGTQ_STATUS_PAGE_RANGE);
        }
    }
    if (active) {
        // every plan-static load of the set-up is issued at once, so that they
        // share one round trip: the K slot lookup recipes (the lane's table
        // copy: + 4 L) and codec pairs of the lane's slots, the query rotation
        // recipe of the lane's codec coordinates 4L..4L+3, and the compact
        // source of the lookup tables
        uint4 km[16];
#pragma unroll
        for (int s = 0; s < 16; ++s) km[s] = __ldg(reinterpret_cast<const uint4*>(&ht->kslot[t][s]));
        const uint4 sp = __ldg(reinterpret_cast<const uint4*>(&ht->slot_pair[t][0]));
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const int j = 4 * lane + i;
            const bool coded = j < n_coded;
            q_pl[i] = coded ? ht->plog2[j] : 0;
            q_src[i] = ht->perm[j];
            q_f[i] = coded ? ht->sign_k[j] * ht->dewhiten[j] : 0.0f;
            q_sc[i] = coded ? ht->inv_sqrt[j] * p.scale_log2 : 0.0f;
        }
        uint32_t* src = reinterpret_cast<uint32_t*>(s_stage);
        const int nw = debug_in_range(p.img_lane + p.img_shared <= kImageMaxWords, tid == 0 ? p.status : nullptr)
                           ? p.img_lane + p.img_shared : 0;
        constexpr int kPerThread = (kImageMaxWords + kWarps * 32 - 1) / (kWarps * 32);
        uint32_t v[kPerThread];
#pragma unroll
        for (int u = 0; u < kPerThread; ++u) {
            const int e = tid + u * kWarps * 32;
            v[u] = e < nw ? __ldg(p.img_src + e) : 0u;
        }
#pragma unroll
        for (int s = 0; s < 16; ++s) {
            ksh[s] = km[s].x;
            kmask[s] = km[s].y;
            kbase[s] = (km[s].z & kSharedTable) ? (km[s].z & ~kSharedTable) : (km[s].z | (4u * lane));
            kwsh[s] = km[s].w;
        }
        slot_pairs[0] = sp.x;
        slot_pairs[1] = sp.y;
        slot_pairs[2] = sp.z;
        slot_pairs[3] = sp.w;
        // the lookup tables: the compact source into the (not yet used)
        // staging region, then 32 copies (one per lane) of every per-lane
        // entry, entry e of lane L at word 32 e + L (a 16-byte store covers 4
        // lanes), and one copy of the shared words
#pragma unroll
        for (int u = 0; u < kPerThread; ++u) {
            const int e = tid + u * kWarps * 32;
            if (e < nw) src[e] = v[u];
        }
        __syncthreads();
        uint4* dst = reinterpret_cast<uint4*>(s_tab);
        for (int i = tid; i < p.img_lane * 8; i += kWarps * 32) {
            const uint32_t x = src[i >> 3];
            dst[i] = make_uint4(x, x, x, x);
        }
        for (int i = tid; i < p.img_shared; i += kWarps * 32) s_tab[32 * p.img_lane + i] = src[p.img_lane + i];
        __syncthreads();  // the source is read before the staging region is reused
    }

    pdl_wait();  // q, the cache and the workspace may belong to the previous kernel
    if (pos_bad && split == 0 && h == 0 && tid == 0 && p.status) {
        atomicOr(p.status, BGTQ_STATUS_APPEND_CAPACITY);
        debug_in_range(false, p.status);  // a new position past the capacity
    }
    // instance 1: the exact logits (q as given . k, on the tensor cores) of
    // the range's window tokens (at most kWinPre), all their key loads in
    // flight at once; the main loop takes them from shared memory.  Warps
    // w0, w0 + stride, ... take the 8-token groups w0, w0 + stride, ...; the
    // new token's key is read as given (its ring slot is being written).
    const bool win_pre = kWinPre1 && p.recent > 0 && active && t_end > wstart;
    auto window_logits = [&](int w0, int stride) {
        const __half* qh = p.q + ((size_t)b * p.H * G + (size_t)h * G) * kD;
        uint2 qo[8];
#pragma unroll
        for (int c = 0; c < 8; ++c) {
            const uint32_t* qw = reinterpret_cast<const uint32_t*>(qh + (size_t)min(g, G - 1) * kD + 16 * c + 2 * t);
            qo[c] = g < G ? make_uint2(__ldg(qw), __ldg(qw + 4)) : make_uint2(0u, 0u);
        }
        const int nwt = min(t_end - wlo, kWinPre);
        // four 8-token groups per round, their key loads issued together
        for (int g0 = w0; 8 * g0 < nwt; g0 += 4 * stride) {
            uint32_t kb[4][8][2];
#pragma unroll
            for (int u = 0; u < 4; ++u) {
                const int tk = min(wlo + 8 * (g0 + u * stride) + g, seq - 1);
                const __half* krow = (p.k_new != nullptr && tk == pos)
                                         ? p.k_new + unit * kD
                                         : p.k_recent + (unit * (size_t)p.recent + (size_t)(tk % p.recent)) * kD;
                const uint32_t* kr = reinterpret_cast<const uint32_t*>(krow + 2 * t);
#pragma unroll
                for (int c = 0; c < 8; ++c) {
                    kb[u][c][0] = __ldcg(kr + 8 * c);
                    kb[u][c][1] = __ldcg(kr + 8 * c + 4);
                }
            }
#pragma unroll
            for (int u = 0; u < 4; ++u) {
                const int grp = g0 + u * stride;
                float s16[4] = {0.0f, 0.0f, 0.0f, 0.0f};
#pragma unroll
                for (int c = 0; c < 8; ++c) {
                    const uint32_t af[4] = {qo[c].x, 0u, qo[c].y, 0u};
                    mma16816(s16, af, kb[u][c][0], kb[u][c][1]);
                }
#pragma unroll
                for (int e = 0; e < 2; ++e) {
                    const int col = 8 * grp + 2 * t + e;
                    if (col < nwt) s_wlog[g][col] = s16[e] * p.scale_log2;
                }
            }
        }
    };
    if (owner) {
        int64_t sl;
        if constexpr (kPaged) {
            sl = sl_new;
            if (sl < 0 && tid == 0 && p.status) atomicOr(p.status, BGTQ_STATUS_PAGE_RANGE);
        } else {
            sl = p.map.slot(b, h, pos);
        }
        if (sl >= 0) append_new_token<BK, BV>(p, el, unit, sl, pos, s_thr, s_enc, warp, lane);  // warps 0, 1
        if (win_pre && warp >= 2) window_logits(warp - 2, kWarps - 2);
        __syncthreads();  // the new token's records are written before any warp stages them
    }
    // the first kStages - 1 tiles of every warp are copied while the queries
    // are rotated
    using SL = StageLayout<BK, BV>;
    uint8_t* st_base = s_stage + warp * (kStages * SL::kBytes);
    const uint32_t st_addr = (uint32_t)__cvta_generic_to_shared(st_base);
    if (active) {
#pragma unroll
        for (int k = 0; k < kStages - 1; ++k) {
            if (k < n_tiles) {
                const int T0 = T0w + k * kStep;
                stage_tile<BK, BV>(st_addr + k * SL::kBytes, kc, vc, kn, vn, kPaged ? s_pslot[warp][k] : tile_slot(T0),
                                   T0, seq, lane);
            }
            cp_async_commit();
        }
    }
    float m_ref = -INFINITY, l_run = 0.0f;  // softmax reference (see kLift, kSlack), sum
    // O^T accumulator: acc[mt][e] = query head 2t + e, codec dim 16 g + 2 mt;
    // acc[mt][2 + e] = the same head, dim 16 g + 2 mt + 1
    float acc[8][4];
#pragma unroll
    for (int i = 0; i < 8; ++i) acc[i][0] = acc[i][1] = acc[i][2] = acc[i][3] = 0.0f;
    if (active) {
    // ---- query heads into the key codec domain: warp w rotates heads
    // kHPW w .. kHPW w + kHPW - 1, lane L holding codec coordinates 4L..4L+3
    // (de-whitening, signs, blockwise Hadamard by shuffles, 1/sqrt(piece),
    // softmax scale, log2 e)
    {
        constexpr int kHPW = (8 + kWarps - 1) / kWarps;
        const __half* qb = p.q + ((size_t)b * p.H * G + (size_t)h * G) * kD;
        float x[kHPW][4];
#pragma unroll
        for (int k = 0; k < kHPW; ++k) {
            const int gg = kHPW * warp + k;
#pragma unroll
            for (int i = 0; i < 4; ++i) x[k][i] = gg < G ? __half2float(qb[(size_t)gg * kD + q_src[i]]) * q_f[i] : 0.0f;
        }
#pragma unroll
        for (int k = 0; k < kHPW; ++k) {
            const int gg = kHPW * warp + k;
            if (gg >= 8) break;
            rotate_warp(x[k], q_pl, lane);
            float a = 0.0f;
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                x[k][i] *= q_sc[i];
                a = fmaxf(a, fabsf(x[k][i]));
            }
#pragma unroll
            for (int o = 16; o >= 1; o >>= 1) a = fmaxf(a, __shfl_xor_sync(0xffffffffu, a, o));
            // Per-head power-of-two scale so the fp16 hi/lo split cannot
            // overflow (whitening moves a key block's scale into the query):
            // max |q| is brought to [2^13, 2^14); logits are scaled back.
            int e = 0;
            if (a > 0.0f && isfinite(a)) frexpf(a, &e);
            e = max(-100, min(100, e));
            const float qs = ldexpf(1.0f, 14 - e);
#pragma unroll
            for (int i = 0; i < 4; ++i) s_q[gg][4 * lane + i] = x[k][i] * qs;
            if (lane == 0) s_qunscale[gg] = ldexpf(1.0f, e - 14);
        }
        // fp16 recent-key buffer: the query heads as given (fp16) as mma A
        // fragments, rows 0..7 = heads (rows 8..15 zero), k-chunk c = dims
        // 16c..16c+15; warp w builds chunks 2w, 2w + 1
        if (kWinLoop && p.recent > 0 && t_end > wstart) {
#pragma unroll
            for (int k = 0; k < 2; ++k) {
                const int c = 2 * warp + k;
                const uint32_t* qw = reinterpret_cast<const uint32_t*>(qb + (size_t)min(g, G - 1) * kD + 16 * c + 2 * t);
                s_qo[c][lane] = g < G ? make_uint2(__ldg(qw), __ldg(qw + 4)) : make_uint2(0u, 0u);
            }
        }
        __syncthreads();  // s_q, s_qunscale, the table image (and a fused step's new token) are complete
        if (win_pre && !owner) {  // (the appending CTA computed them during its append)
            window_logits(warp, kWarps);
            __syncthreads();
        }
    }
    const float q_unscale = s_qunscale[g];
    uint32_t qa[8][4];
#pragma unroll
    for (int c = 0; c < 8; ++c) {
        const int m0 = (slot_pairs[c >> 1] >> (16 * (c & 1))) & 255;
        const int m1 = (slot_pairs[c >> 1] >> (16 * (c & 1) + 8)) & 255;
        const float x0 = s_q[g][(2 * m0) & (kD - 1)], x1 = s_q[g][(2 * m0 + 1) & (kD - 1)];
        const float y0 = s_q[g][(2 * m1) & (kD - 1)], y1 = s_q[g][(2 * m1 + 1) & (kD - 1)];
        const bool v0 = 2 * m0 < n_coded, v1 = 2 * m1 < n_coded;
        split_hilo(v0 ? x0 : 0.0f, v0 ? x1 : 0.0f, qa[c][0], qa[c][1]);
        split_hilo(v1 ? y0 : 0.0f, v1 ? y1 : 0.0f, qa[c][2], qa[c][3]);
    }
    // value tables: the lane's copy of the width-BV pair table, or of the
    // width-4 single table
    const uint32_t vbase = (BV <= kPairTableMaxW ? (1u << (2 * BV)) << 7 : (uint32_t)single_base(4) << 7) | (4u * lane);

    // ---- main loop: 16-token tiles, operands of the next tile loaded while
    // the current one is decoded (ping-pong register buffers).  kWin: the
    // tile reaches into the fp16 recent-key buffer.
    auto process = [&](const TileRegs<BK, BV>& tr, int T0, auto win) {
        constexpr bool kWin = decltype(win)::value;
        // recent-key buffer tile: its fp16 keys, as mma B fragments of ring
        // slot pos mod W (token row g of 8-token group nt).  The fast
        // instance fetches them first, so that the fetch overlaps the
        // packed-key decode below; the general one (no registers to spare)
        // right before use.
        uint32_t kb[2][8][2];
        auto load_kb = [&]() {
#pragma unroll
            for (int nt = 0; nt < 2; ++nt) {
                const int tk = min(max(T0 + 8 * nt + g, wstart), seq - 1);
                const uint32_t* kr = reinterpret_cast<const uint32_t*>(
                    p.k_recent + (unit * (size_t)p.recent + (size_t)(tk % p.recent)) * kD + 2 * t);
#pragma unroll
                for (int c = 0; c < 8; ++c) {
                    kb[nt][c][0] = __ldcg(kr + 8 * c);
                    kb[nt][c][1] = __ldcg(kr + 8 * c + 4);
                }
            }
        };
        if constexpr (kWin && NW != 16) load_kb();
        float sacc[2][4];
#pragma unroll
        for (int nt = 0; nt < 2; ++nt) sacc[nt][0] = sacc[nt][1] = sacc[nt][2] = sacc[nt][3] = 0.0f;
        const uint64_t wl[2] = {kwin_lo<BK>(tr.kw[0]), kwin_lo<BK>(tr.kw[1])};
        const uint64_t wh[2] = {kwin_hi<BK>(tr.kw[0]), kwin_hi<BK>(tr.kw[1])};
        s_chunk<NW, 0>(sacc, qa, wl, wh, ksh, kmask, kbase, kwsh, s_tab);
        s_chunk<NW, 1>(sacc, qa, wl, wh, ksh, kmask, kbase, kwsh, s_tab);
        s_chunk<NW, 2>(sacc, qa, wl, wh, ksh, kmask, kbase, kwsh, s_tab);
        s_chunk<NW, 3>(sacc, qa, wl, wh, ksh, kmask, kbase, kwsh, s_tab);
        s_chunk<NW, 4>(sacc, qa, wl, wh, ksh, kmask, kbase, kwsh, s_tab);
        s_chunk<NW, 5>(sacc, qa, wl, wh, ksh, kmask, kbase, kwsh, s_tab);
        s_chunk<NW, 6>(sacc, qa, wl, wh, ksh, kmask, kbase, kwsh, s_tab);
        s_chunk<NW, 7>(sacc, qa, wl, wh, ksh, kmask, kbase, kwsh, s_tab);
        // logits (log2 domain) of head g for tokens T0 + 8 nt + 2 t + e
        float lg[2][2];
#pragma unroll
        for (int nt = 0; nt < 2; ++nt)
#pragma unroll
            for (int e = 0; e < 2; ++e) {
                const int tok = T0 + 8 * nt + 2 * t + e;
                float v = (sacc[nt][e] + sacc[nt][2 + e]) * (tr.rk[nt][e] * q_unscale);
                if constexpr (kWinPre1) {
                    if (tok >= wstart && tok < t_end) v = s_wlog[g][(tok - wlo) & (kWinPre - 1)];
                }
                lg[nt][e] = tok < t_end ? v : -INFINITY;
            }
        if constexpr (kWin) {
            // the tokens of the tile inside the fp16 recent-key buffer take
            // their logits from their exact keys (q as given . k, on the
            // tensor cores)
            if constexpr (NW == 16) load_kb();
            float s16[2][4];
#pragma unroll
            for (int nt = 0; nt < 2; ++nt) s16[nt][0] = s16[nt][1] = s16[nt][2] = s16[nt][3] = 0.0f;
#pragma unroll
            for (int c = 0; c < 8; ++c) {
                const uint2 a = s_qo[c][lane];
                const uint32_t af[4] = {a.x, 0u, a.y, 0u};
#pragma unroll
                for (int nt = 0; nt < 2; ++nt) mma16816(s16[nt], af, kb[nt][c][0], kb[nt][c][1]);
            }
#pragma unroll
            for (int nt = 0; nt < 2; ++nt)
#pragma unroll
                for (int e = 0; e < 2; ++e) {
                    const int tok = T0 + 8 * nt + 2 * t + e;
                    if (tok >= wstart && tok < t_end) lg[nt][e] = s16[nt][e] * p.scale_log2;
                }
        }
        float mx = -INFINITY;
#pragma unroll
        for (int nt = 0; nt < 2; ++nt) mx = fmaxf(mx, fmaxf(lg[nt][0], lg[nt][1]));
        mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 1));
        mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 2));
        if (__any_sync(0xffffffffu, mx > m_ref + kSlack)) {
            const float ref = mx > m_ref + kSlack ? mx + kLift : m_ref;
            const float alpha = fast_exp2(m_ref - ref);
            l_run *= alpha;
            // the accumulator of lane (g, t) holds query heads 2t and 2t + 1:
            // their factors come from the lanes of those heads
            const float a0 = __shfl_sync(0xffffffffu, alpha, 8 * t);
            const float a1 = __shfl_sync(0xffffffffu, alpha, 8 * t + 4);
#pragma unroll
            for (int i = 0; i < 8; ++i) {
                acc[i][0] *= a0;
                acc[i][1] *= a1;
                acc[i][2] *= a0;
                acc[i][3] *= a1;
            }
            m_ref = ref;
        }
        float pr[2][2];
#pragma unroll
        for (int nt = 0; nt < 2; ++nt)
#pragma unroll
            for (int e = 0; e < 2; ++e) {
                pr[nt][e] = fast_exp2(lg[nt][e] - m_ref);
                l_run += pr[nt][e];
            }
        // P' = p * rho_V of head g for tokens 2t, 2t+1 (b0) and 8+2t, 9+2t
        // (b1): the B fragment of the P.V product, split hi + lo
        uint32_t pb[2][2];
        split_hilo(pr[0][0] * tr.rv[0][0], pr[0][1] * tr.rv[0][1], pb[0][0], pb[1][0]);
        split_hilo(pr[1][0] * tr.rv[1][0], pr[1][1] * tr.rv[1][1], pb[0][1], pb[1][1]);
        pv_mtile<BV, 0>(acc, pb, tr.vw, vbase, s_tab);
        pv_mtile<BV, 1>(acc, pb, tr.vw, vbase, s_tab);
        pv_mtile<BV, 2>(acc, pb, tr.vw, vbase, s_tab);
        pv_mtile<BV, 3>(acc, pb, tr.vw, vbase, s_tab);
        pv_mtile<BV, 4>(acc, pb, tr.vw, vbase, s_tab);
        pv_mtile<BV, 5>(acc, pb, tr.vw, vbase, s_tab);
        pv_mtile<BV, 6>(acc, pb, tr.vw, vbase, s_tab);
        pv_mtile<BV, 7>(acc, pb, tr.vw, vbase, s_tab);
    };

    auto step = [&](int k, auto win) {
        const int kn_ = k + kStages - 1;
        if (kn_ < n_tiles) {
            const int T0 = T0w + kn_ * kStep;
            stage_tile<BK, BV>(st_addr + (kn_ % kStages) * SL::kBytes, kc, vc, kn, vn,
                               kPaged ? s_pslot[warp][kn_] : tile_slot(T0), T0, seq, lane);
        }
        cp_async_commit();
        cp_async_wait<kStages - 1>();
        __syncwarp();
        TileRegs<BK, BV> tr;
        tr.read(st_base + (k % kStages) * SL::kBytes, g, t);
        process(tr, T0w + k * kStep, win);
        __syncwarp();  // the stage is refilled next
    };
    // the tiles that reach into the fp16 recent-key buffer are the warp's
    // last few; the loop over the others carries no trace of the buffer
    int n_fast = n_tiles;
    if (kWinLoop && p.recent > 0) {
        const int d = wstart - kTile - T0w;
        n_fast = d < 0 ? 0 : min(n_tiles, d / kStep + 1);
    }
    for (int k = 0; k < n_fast; ++k) step(k, BoolTag<false>{});
    if constexpr (kWinLoop)
        for (int k = n_fast; k < n_tiles; ++k) step(k, BoolTag<true>{});
    cp_async_wait<0>();
    }  // active

    // ---- the warp's partial (m, l, acc) of its 8 query heads -> s_wp[warp]
    __syncthreads();  // every warp is done with the tables
    l_run += __shfl_xor_sync(0xffffffffu, l_run, 1);
    l_run += __shfl_xor_sync(0xffffffffu, l_run, 2);
    if (t == 0) {
        s_wp[warp][g][0] = m_ref;
        s_wp[warp][g][1] = l_run;
    }
#pragma unroll
    for (int mt = 0; mt < 8; ++mt)
#pragma unroll
        for (int e = 0; e < 2; ++e) {
            s_wp[warp][2 * t + e][2 + 16 * g + 2 * mt] = acc[mt][e];
            s_wp[warp][2 * t + e][2 + 16 * g + 2 * mt + 1] = acc[mt][2 + e];
        }

    // ---- CTA merge: thread tid merges query head tid / 16, dims
    // 8 (tid % 16) .. + 7, over the 4 warps -> s_cp
    static_assert(kWarps * 32 == 16 * 8, "CTA merge: 16 threads per head, 8 dims each");
    __syncthreads();
    {
        const int hh = tid >> 4, d0 = 8 * (tid & 15);
        float mw[kWarps], fw[kWarps];
        float M = -INFINITY, L = 0.0f;
#pragma unroll
        for (int w = 0; w < kWarps; ++w) {
            mw[w] = s_wp[w][hh][0];
            M = fmaxf(M, mw[w]);
        }
#pragma unroll
        for (int w = 0; w < kWarps; ++w) {
            fw[w] = mw[w] == -INFINITY ? 0.0f : exp2f(mw[w] - M);
            L += s_wp[w][hh][1] * fw[w];
        }
        float o[8];
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            o[i] = 0.0f;
#pragma unroll
            for (int w = 0; w < kWarps; ++w) o[i] += fw[w] * s_wp[w][hh][2 + d0 + i];
        }
#pragma unroll
        for (int i = 0; i < 8; ++i) s_cp[hh][2 + d0 + i] = o[i];
        if ((tid & 15) == 0) {
            s_cp[hh][0] = M;
            s_cp[hh][1] = L;
        }
    }

    // ---- cluster merge: CTA rank r reduces query heads r, r + kCluster, ...
    // over the kCluster CTA partials of the cluster, read through distributed
    // shared memory (lane c < kCluster takes the (m, l) of CTA c; thread tid
    // holds dim tid of acc)
    constexpr int kHeadsPerCta = (8 + kCluster - 1) / kCluster;
    static_assert(kCluster <= 32 && kWarps * 32 >= kD, "cluster merge layout");
    cluster.sync();
    const size_t max_clusters = (size_t)p.n_split / kCluster;
    float* cpart_base = p.part + unit * max_clusters * (size_t)G * kPartStride;
    float Mc[kHeadsPerCta], Lc[kHeadsPerCta], Oc[kHeadsPerCta];
#pragma unroll
    for (int j = 0; j < kHeadsPerCta; ++j) {
        const int hh = crank + j * kCluster;
        Mc[j] = -INFINITY;
        Lc[j] = 0.0f;
        Oc[j] = 0.0f;
        if (hh >= G) continue;
        float mi = -INFINITY, li = 0.0f;
        if (lane < kCluster) {
            const float* src = cluster.map_shared_rank(&s_cp[hh][0], lane);
            mi = src[0];
            li = src[1];
        }
        float M = mi;
#pragma unroll
        for (int o = 16; o >= 1; o >>= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, o));
        const float fi = mi == -INFINITY ? 0.0f : exp2f(mi - M);
        float L = li * fi;
#pragma unroll
        for (int o = 16; o >= 1; o >>= 1) L += __shfl_xor_sync(0xffffffffu, L, o);
        float O = 0.0f;
        if (tid < kD) {
            float x[kCluster];
#pragma unroll
            for (int c = 0; c < kCluster; ++c) x[c] = *cluster.map_shared_rank(&s_cp[hh][2 + tid], c);
#pragma unroll
            for (int c = 0; c < kCluster; ++c) O += __shfl_sync(0xffffffffu, fi, c) * x[c];
        }
        Mc[j] = M;
        Lc[j] = L;
        Oc[j] = O;
    }
    cluster_arrive();  // this CTA has finished reading the other CTAs' partials
#pragma unroll
    for (int j = 0; j < kHeadsPerCta; ++j) {
        const int r = crank + j * kCluster;
        if (r >= G) continue;
        float* dst = cpart_base + ((size_t)cid * G + r) * kPartStride;
        if (tid < kD) dst[2 + tid] = Oc[j];
        if (tid == 0) {
            dst[0] = Mc[j];
            dst[1] = Lc[j];
        }
        __syncthreads();  // the partial is written before thread 0 releases it
        if (tid == 0) {
            const unsigned prev = ticket_acq_rel(p.count + unit * G + r);
            s_last = (prev == (unsigned)(n_clusters - 1)) ? 1 : 0;
        }
        __syncthreads();  // thread 0's acquire is ordered before the loads below
        if (!s_last) continue;
        // ---- last cluster partial of query head r: warp w merges the
        // partials of clusters w, w + kWarps, ... (one batch of independent
        // loads; lane holds dims lane + 32 i) into the free per-warp region,
        // then warp 0 merges the kWarps results
        constexpr int kPerWarp = (kMaxClusters + kWarps - 1) / kWarps;
        float M = -INFINITY, L = 0.0f, O[4] = {0.0f, 0.0f, 0.0f, 0.0f};
        float sgn[4];  // value rotation signs of the lane's output dims, fetched with the partials
#pragma unroll
        for (int i = 0; i < 4; ++i) sgn[i] = warp == 0 ? __ldg(&ht->sign_v[lane + 32 * i]) * p.v_inv_sqrt : 0.0f;
        {
            float mc[kPerWarp], lc[kPerWarp], oc[kPerWarp][4];
#pragma unroll
            for (int jj = 0; jj < kPerWarp; ++jj) {
                const int c = warp + kWarps * jj;
                mc[jj] = -INFINITY;
                lc[jj] = 0.0f;
                oc[jj][0] = oc[jj][1] = oc[jj][2] = oc[jj][3] = 0.0f;
                if (c < n_clusters) {
                    const float* src = cpart_base + ((size_t)c * G + r) * kPartStride;
                    mc[jj] = __ldcg(src);
                    lc[jj] = __ldcg(src + 1);
#pragma unroll
                    for (int i = 0; i < 4; ++i) oc[jj][i] = __ldcg(src + 2 + lane + 32 * i);
                }
            }
#pragma unroll
            for (int jj = 0; jj < kPerWarp; ++jj) M = fmaxf(M, mc[jj]);
#pragma unroll
            for (int jj = 0; jj < kPerWarp; ++jj) {
                const float f = mc[jj] == -INFINITY ? 0.0f : exp2f(mc[jj] - M);
                L += lc[jj] * f;
#pragma unroll
                for (int i = 0; i < 4; ++i) O[i] += oc[jj][i] * f;
            }
        }
        float* sw = &s_wp[warp][0][0];
        if (lane == 0) {
            sw[0] = M;
            sw[1] = L;
        }
#pragma unroll
        for (int i = 0; i < 4; ++i) sw[2 + lane + 32 * i] = O[i];
        __syncthreads();
        if (warp == 0) {
            float mw[kWarps];
            float Mt = -INFINITY;
#pragma unroll
            for (int w = 0; w < kWarps; ++w) {
                mw[w] = s_wp[w][0][0];
                Mt = fmaxf(Mt, mw[w]);
            }
            L = 0.0f;
            O[0] = O[1] = O[2] = O[3] = 0.0f;
#pragma unroll
            for (int w = 0; w < kWarps; ++w) {
                const float f = mw[w] == -INFINITY ? 0.0f : exp2f(mw[w] - Mt);
                L += s_wp[w][0][1] * f;
#pragma unroll
                for (int i = 0; i < 4; ++i) O[i] += s_wp[w][0][2 + lane + 32 * i] * f;
            }
        }
        __syncthreads();  // the per-warp region is read before a next head reuses it
        if (warp != 0) continue;
        // inverse value rotation (Hadamard-128, 1/sqrt(128), signs): stages
        // 1..16 by shuffles, 32 and 64 between the lane's four dims
        float v[4];
#pragma unroll
        for (int i = 0; i < 4; ++i) v[i] = O[i] / L;
#pragma unroll
        for (int hh = 1; hh < 32; hh <<= 1) {
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                const float o = __shfl_xor_sync(0xffffffffu, v[i], hh);
                v[i] = (lane & hh) ? o - v[i] : v[i] + o;
            }
        }
        {
            const float a0 = v[0] + v[1], a1 = v[0] - v[1], a2 = v[2] + v[3], a3 = v[2] - v[3];
            v[0] = a0 + a2;
            v[2] = a0 - a2;
            v[1] = a1 + a3;
            v[3] = a1 - a3;
        }
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const int d = lane + 32 * i;
            const float val = v[i] * sgn[i];
            const size_t o = ((size_t)b * p.H * G + (size_t)h * G + r) * kD + d;
            if (p.out_dtype) static_cast<float*>(p.out)[o] = val;
            else static_cast<__half*>(p.out)[o] = __float2half_rn(val);
        }
        if (lane == 0) p.count[unit * G + r] = 0;
    }
    cluster_wait();  // no CTA leaves while another may still read its partials
}

// The dynamic shared memory of the three instances of decode_kernel<BK, BV>
// of one paging mode is raised above the 48 KB default once per device, to
// the size with the largest lookup tables.
template <int BK, int BV, bool kPaged>
cudaError_t ensure_smem_attr() {
    static std::mutex mu;
    static bool done[64] = {false};
    int dev = 0;
    cudaGetDevice(&dev);
    if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
    std::lock_guard<std::mutex> lock(mu);
    if (done[dev]) return cudaSuccess;
    const int bytes = decode_smem_bytes<BK, BV>(kWMax);
    cudaError_t e = cudaFuncSetAttribute(decode_kernel<BK, BV, 0, kPaged>, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
    if (e == cudaSuccess)
        e = cudaFuncSetAttribute(decode_kernel<BK, BV, 1, kPaged>, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
    if (e == cudaSuccess)
        e = cudaFuncSetAttribute(decode_kernel<BK, BV, 2, kPaged>, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
    if (e == cudaSuccess) done[dev] = true;
    return e;
}

template <int BK, int BV>
cudaLaunchConfig_t launch_config(dim3 grid, cudaStream_t s, int ws, cudaLaunchAttribute* attr /*[2]*/) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = dim3(kWarps * 32, 1, 1);
    cfg.dynamicSmemBytes = decode_smem_bytes<BK, BV>(ws);
    cfg.stream = s;
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = kCluster;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[1].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 2;
    return cfg;
}

template <int BK, int BV, bool kPaged>
cudaError_t launch_t(DecodeParams p, dim3 grid, cudaStream_t s, int kind) {
    cudaError_t e = ensure_smem_attr<BK, BV, kPaged>();
    if (e != cudaSuccess) return e;
    const int ws = p.img_ws;
    p.img_bytes = decode_table_bytes(ws);
    cudaLaunchAttribute attr[2];
    cudaLaunchConfig_t cfg = launch_config<BK, BV>(grid, s, ws, attr);
    if (kind == 2) return cudaLaunchKernelEx(&cfg, decode_kernel<BK, BV, 2, kPaged>, p);
    if (kind == 1) return cudaLaunchKernelEx(&cfg, decode_kernel<BK, BV, 1, kPaged>, p);
    return cudaLaunchKernelEx(&cfg, decode_kernel<BK, BV, 0, kPaged>, p);
}

}  // namespace
}  // namespace bgtq
