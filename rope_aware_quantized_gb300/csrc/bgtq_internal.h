// Library-internal types shared by the host planner and the CUDA kernels.
#pragma once

#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

#include <string>
#include <vector>

#include "bgtq.h"

namespace bgtq {

constexpr int kD = 128;      // head dim
constexpr int kNB = 64;      // RoPE 2-D blocks per key
constexpr int kWMax = 8;     // widest code
constexpr int kPairMaxW = 5; // widest code decoded through the pair table

// Pair table: entry (4^w + f) holds half2(c_w[f & (2^w-1)], c_w[f >> w]) for
// w = 0..kPairMaxW, so a pre-shifted field f<<2 is OR-ed with (4^w)<<2.
constexpr int kPairLutWords = 1 << (2 * kPairMaxW + 1);
// Single table: entry (2^w + c) holds c_w[c] (fp16 bits) for w = 0..8.
constexpr int kSingleLutHalves = 1 << (kWMax + 1);

// Shared-memory image of the decode tables (32-bit words), copied verbatim
// by every decode CTA.  Arranged so that the lanes of a warp rarely collide
// on a bank:
//   [0, 2048)       pair tables of widths 0..5, shared by all lanes (entry 4^w + f)
//   [2048, 4096)    8 copies of the width-4 pair table, one per token lane g
//                   (entry 256 + f of copy g at 2048 + 8 f + g)
//   [4096, 8192)    per-lane copies of the pair tables of widths 0..3
//                   (entry e of lane L at 4096 + 32 e + L)
//   [8192, 10240)   8 copies of the single-entry table by token lane g, as
//                   fp16 halves (entry 2^w + c of copy g at half 8 (2^w + c) + g)
constexpr int kImgG4 = 2048;
constexpr int kImgPriv = 4096;
constexpr int kImgSingle = 8192;
constexpr int kImgWords = 10240;

// How decode lane (g, t) extracts and looks up one K slot: the 64-bit window
// is shifted right by `sh` (slot 0: its word is shifted left by `sh`), masked
// with `mask` and OR-ed with base + (mult & 255) * lane + (mult >> 8) * g.
struct SlotMeta {
    uint32_t sh, mask, base, mult;
};

// Per-head device tables.  All arrays are in codec order unless noted.
struct HeadTab {
    int32_t n_coded;
    uint32_t wide_mask;       // decode: slots decoded through the single table
    int32_t pad[2];
    uint8_t perm[kD];         // codec index -> original dim
    uint8_t width[kD];        // code width per codec index (0 past n_coded)
    uint8_t plog2[kD];        // log2 of the rotation piece size (0 past n_coded)
    uint8_t slot_pair[4][16]; // decode lane layout: codec pair per (lane, slot)
    uint8_t slot_w[4][16];    // width of that pair
    uint8_t slot_sh[4][16];   // field shift inside the slot's 64-bit window
    uint16_t pair_bit[kNB];   // absolute bit position of codec pair m in the K record
    float whiten[kD];
    float dewhiten[kD];
    float inv_sqrt[kD];
    float sign_k[kD];
    float sign_v[kD];
    SlotMeta kmeta[4][16];    // decode: lookup recipe of (lane t, slot)
};

static_assert(offsetof(HeadTab, kmeta) % 16 == 0 && sizeof(HeadTab) % 16 == 0,
              "decode loads the lookup recipes with 16-byte loads");

struct DevTables {
    HeadTab* heads = nullptr;     // [H]
    float* cent = nullptr;        // [9][256] centroids (fp16-exact floats)
    float* thr = nullptr;         // [9][256] thresholds (first 2^w - 1 used)
    uint32_t* pair_lut = nullptr; // [kPairLutWords]
    uint16_t* single_lut = nullptr; // [kSingleLutHalves]
    uint32_t* dec_image = nullptr;  // [kImgWords] decode shared-memory image
};

// Where the records of (sequence b, head h, position pos) live: token slot
// (b H + h) capacity + pos of a contiguous cache, or (page H + h) P + pos mod P
// of a paged one (page = page_table[b][pos / P]).  K record, norms: index
// slot; V pair record of the pair holding pos: index slot / 2 (P and the
// capacity are even, so a pair never straddles two pages).
struct CacheMap {
    const int32_t* page_table;  // [B][max_pages], nullptr: contiguous
    int64_t cap;                // positions per sequence (capacity = max_pages * P when paged)
    int64_t max_pages, n_pages;
    int H, lp;                  // lp = log2 P (paged)
#ifdef __CUDACC__
    // -1 when the page_table entry is outside [0, n_pages)
    __device__ __forceinline__ int64_t slot(int b, int h, int64_t pos) const {
        if (!page_table) return ((int64_t)b * H + h) * cap + pos;
        const int32_t pg = page_table[(int64_t)b * max_pages + (pos >> lp)];
        if (pg < 0 || (int64_t)pg >= n_pages) return -1;
        return (((int64_t)pg * H + h) << lp) + (pos & ((((int64_t)1) << lp) - 1));
    }
#endif
};

cudaError_t launch_prefill(const bgtq_plan& pl, cudaStream_t s, const void* q, const void* k, const void* v,
                           int batch, int t, const bgtq_cache& c, void* out, int out_dtype, float scale,
                           int32_t* status);

// Host checks of a cache descriptor (buffers, alignment, capacity, the
// recent-key buffer, paging); sets the thread's error message.
int check_cache(const bgtq_plan* p, const bgtq_cache* c);

inline CacheMap make_cache_map(const bgtq_cache& c, int H) {
    CacheMap m;
    m.page_table = c.page_table;
    m.cap = c.capacity;
    m.max_pages = c.page_table ? c.max_pages : 1;
    m.n_pages = c.page_table ? c.n_pages : 1;
    m.H = H;
    m.lp = 0;
    if (c.page_table)
        while (((int64_t)1 << m.lp) < c.page_tokens) ++m.lp;
    return m;
}

}  // namespace bgtq

struct bgtq_plan {
    int H = 0, G = 0, bits_per_key = 0, bk = 0, bv = 0, rope_layout = 0, flags = 0;
    uint64_t seed = 0;
    int device = -1, num_sms = 0;
    std::vector<bgtq::HeadTab> heads;
    std::vector<float> cent[bgtq::kWMax + 1];
    std::vector<float> thr[bgtq::kWMax + 1];
    std::vector<uint32_t> pair_lut;
    std::vector<uint16_t> single_lut;
    std::vector<uint32_t> dec_image;
    // inspection copies (bgtq_plan_get_head)
    std::vector<std::vector<int8_t>> sign_k8, sign_v8;
    std::vector<std::vector<uint8_t>> piece;
    std::vector<std::vector<uint16_t>> slot_off;
    bgtq::DevTables dev;
};

namespace bgtq {

int set_error(int code, const char* fmt, ...);

// Kernel launchers (defined in the .cu files).  They only enqueue work.
cudaError_t launch_quantize_append(const bgtq_plan& p, cudaStream_t s, const void* k, const void* v, int batch,
                                   int t_new, const int32_t* pos_start, const bgtq_cache& c, int32_t* status);
cudaError_t launch_dequant(const bgtq_plan& p, cudaStream_t s, const bgtq_cache& c, int batch, int b, int head,
                           int64_t t0, int64_t t1, float* k_out, float* v_out, int codec_domain);

cudaError_t launch_logit_mae(const bgtq_plan& p, cudaStream_t s, const void* q, const void* k, const bgtq_cache& c,
                             int64_t t, int batch, float scale, float* out);

struct SplitPlan {
    int n_split = 1;
    int tokens_per_split = 64;
};
SplitPlan decode_split(const bgtq_plan& p, int batch, int64_t max_len);
size_t decode_workspace_bytes(const bgtq_plan& p, int batch, const SplitPlan& sp);
// bytes of per-(sequence, KV head, query head) arrival counters at the front
// of the decode workspace (they must be zero before a call; calls leave them zero)
size_t decode_counter_bytes(const bgtq_plan& p, int batch);
// k_new/v_new/pos_new non-null: the fused step (append one token per
// sequence, then attend); null: attention only.
cudaError_t launch_decode(const bgtq_plan& p, cudaStream_t s, const void* q, const bgtq_cache& c,
                          const int32_t* seq_lens, int batch, const SplitPlan& sp, void* out, int out_dtype,
                          float scale, void* ws, int32_t* status, const void* k_new = nullptr,
                          const void* v_new = nullptr, const int32_t* pos_new = nullptr);

}  // namespace bgtq
