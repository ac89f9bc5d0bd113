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
constexpr int kPairMaxW = 5; // widest value code of a plan

// Decode lookup tables in shared memory.  Tables of widths up to 6 hold one
// copy of every entry per lane (entry e of lane L is word 32 e + L), so the 32
// lookups of a warp instruction fall on 32 distinct banks whatever the codes:
//   entries [0, 128): pair tables of widths 0..3; entry 4^w + f holds the fp16
//     pair (c_w[f mod 2^w], c_w[f >> w]) (entry 0 is zero)
//   entries single_base(w) + c, widths 4..6: c_w[c] in both halves; every
//     base is a multiple of 2^w, so an entry address is (c << 7) | (base << 7) | 4 L.
// The rare widths 7 and 8 have one shared copy after the per-lane region
// (word shared_word(w) + c, both halves), looked up with a 4-byte stride.
constexpr int kPairEntries = 128;
constexpr int kPairTableMaxW = 3;   // widths decoded as pairs (one lookup per two codes)
constexpr int kLaneTableMaxW = 6;   // widest code with per-lane copies
__host__ __device__ constexpr int single_base(int w) { return w == 4 ? 128 : w == 5 ? 160 : 192; }
// per-lane entries for codes up to width ws
__host__ __device__ constexpr int lane_entries(int ws) { return ws <= 3 ? 128 : ws == 4 ? 144 : ws == 5 ? 192 : 256; }
// shared words for codes up to width ws (width 8 at word 0, width 7 after it)
__host__ __device__ constexpr int shared_words(int ws) { return ws <= 6 ? 0 : ws == 7 ? 128 : 384; }
__host__ __device__ constexpr int shared_word(int w, int ws) { return w == 8 ? 0 : (ws >= 8 ? 256 : 0); }
constexpr int kImageMaxWords = 256 + 384;  // lane_entries(8) + shared_words(8): words of the compact source
// bytes of the table region for codes up to width ws
__host__ __device__ constexpr int image_bytes(int ws) { return lane_entries(ws) * 128 + shared_words(ws) * 4; }

// Lookup recipe of K slot (lane t, slot s): the slot's 64-bit window (slots
// 0..7: the lane slice shifted left by 7 bits; slots 8..15: the slice's upper
// two words, or its two words, or its one word) shifted right by `sh` puts
// the slot's first code at bit 7 (per-lane tables) or bit 2 (shared tables);
// `mask` keeps the field (pair table: both codes, 2w bits; single table: the
// first code, w bits) and `base` is the table's byte base, to which the lane
// adds 4 L unless bit 31 (kSharedTable) is set.  Single-table slots (w >= 4)
// look up the second code w bits higher (wsh = w); pair-table slots have
// wsh = 0.
struct KSlot {
    uint32_t sh, mask, base, wsh;
};
constexpr uint32_t kSharedTable = 0x80000000u;

// Per-head device tables.  All arrays are in codec order unless noted.
struct HeadTab {
    int32_t n_coded;
    int32_t n_wide;           // decode: leading slots (in width order 0, 8, 1, 9, ...) that may hold w >= 4
    int32_t max_w;            // widest key code
    int32_t pad;
    uint8_t perm[kD];         // codec index -> original dim
    uint8_t width[kD];        // code width per codec index (0 past n_coded)
    uint8_t plog2[kD];        // log2 of the rotation piece size (0 past n_coded)
    uint8_t slot_pair[4][16]; // decode lane layout: codec pair per (lane, slot)
    uint16_t pair_bit[kNB];   // absolute bit position of codec pair m in the K record
    float whiten[kD];
    float dewhiten[kD];
    float inv_sqrt[kD];
    float sign_k[kD];
    float sign_v[kD];
    KSlot kslot[4][16];       // decode: lookup recipe of (lane t, slot)
};

static_assert(offsetof(HeadTab, kslot) % 16 == 0 && sizeof(HeadTab) % 16 == 0,
              "decode loads the lookup recipes with 16-byte loads");

struct DevTables {
    HeadTab* heads = nullptr;     // [H]
    float* cent = nullptr;        // [9][256] centroids (fp16-exact floats)
    float* thr = nullptr;         // [9][256] thresholds (first 2^w - 1 used)
    uint32_t* img_src = nullptr;  // [kImageMaxWords] decode tables: per-lane entries, then shared words
    uint32_t* cells = nullptr;    // code-search cell tables (layout: kCellHdr)
};

// Code-search cell tables of the bulk encoder (built with the codebooks).
// Words: for each width w = 0..8 four words (a, b, s as float bits, index of
// the width's first entry), then the entries, two words each (threshold as
// float bits, +inf if none; number of thresholds in the cells below).  The
// cell of a quotient u at width w is round(s * sat(a u + b)), found as the
// low bits of fma(sat(fma(u, a, b)), s, 1.5 * 2^23).
constexpr int kCellHdr = 4 * (kWMax + 1);
constexpr int kCellMaxEntries = 1536;
constexpr uint32_t kCellMagicBits = 0x4B400000u;  // bits of 1.5 * 2^23

// Where the records of (sequence b, head h, position pos) live: token slot
// (b H + h) capacity + pos of a contiguous cache, or (page H + h) P + pos mod P
// of a paged one (page = page_table[b][pos / P]).  K record, norms: index
// slot; V pair record of the pair holding pos: index slot / 2 (P and the
// capacity are even, so a pair never straddles two pages).
#ifdef __CUDACC__
// Range checks of the BGTQ_DEBUG_BOUNDS build: a failed check ORs
// BGTQ_STATUS_BOUNDS into the launch's status word and its caller skips the
// access (no trap).  In the default build every check is `true` and the
// condition compiles away.
__device__ __forceinline__ bool debug_in_range(bool ok, int32_t* status) {
#ifdef BGTQ_DEBUG_BOUNDS
    if (!ok && status) atomicOr(status, BGTQ_STATUS_BOUNDS);
    return ok;
#else
    (void)ok;
    (void)status;
    return true;
#endif
}
#endif

struct CacheMap {
    const int32_t* page_table;  // [B][max_pages], nullptr: contiguous
    int64_t cap;                // positions per sequence (capacity = max_pages * P when paged)
    int64_t max_pages, n_pages;
    int H, lp;                  // lp = log2 P (paged)
    int batch;                  // sequences of the launch
    int64_t n_slots;            // record slots: batch H cap, or n_pages H P when paged
    int32_t* status;            // where a failed range check is reported
#ifdef __CUDACC__
    // -1 when the page_table entry is outside [0, n_pages) (and, in the
    // BGTQ_DEBUG_BOUNDS build, when b, h, pos or the slot is out of range)
    __device__ __forceinline__ int64_t slot(int b, int h, int64_t pos) const {
        if (!debug_in_range(b >= 0 && b < batch && h >= 0 && h < H && pos >= 0 && pos < cap, status)) return -1;
        if (!page_table) return ((int64_t)b * H + h) * cap + pos;
        const int32_t pg = page_table[(int64_t)b * max_pages + (pos >> lp)];
        if (pg < 0 || (int64_t)pg >= n_pages) {
            debug_in_range(false, status);
            return -1;
        }
        const int64_t sl = (((int64_t)pg * H + h) << lp) + (pos & ((((int64_t)1) << lp) - 1));
        return debug_in_range(sl < n_slots, status) ? sl : -1;
    }
#endif
};

cudaError_t launch_prefill(const bgtq_plan& pl, cudaStream_t s, const void* q, const void* k, const void* v,
                           int batch, int t, const bgtq_cache& c, void* out, int out_dtype, float scale,
                           int32_t* status);
size_t prefill_chunk_workspace_bytes(const bgtq_plan& pl, int batch, int64_t max_prefix);
cudaError_t launch_prefill_chunk(const bgtq_plan& pl, cudaStream_t s, const void* q, const void* k, const void* v,
                                 int batch, int c, const int32_t* pos_start, int64_t max_prefix, const bgtq_cache& cache,
                                 void* out, int out_dtype, float scale, void* ws, int32_t* status);

// Host checks of a cache descriptor (buffers, alignment, capacity, the
// recent-key buffer, paging); sets the thread's error message.
int check_cache(const bgtq_plan* p, const bgtq_cache* c);

inline CacheMap make_cache_map(const bgtq_cache& c, int H, int batch, int32_t* status) {
    CacheMap m;
    m.page_table = c.page_table;
    m.cap = c.capacity;
    m.max_pages = c.page_table ? c.max_pages : 1;
    m.n_pages = c.page_table ? c.n_pages : 1;
    m.H = H;
    m.lp = 0;
    if (c.page_table)
        while (((int64_t)1 << m.lp) < c.page_tokens) ++m.lp;
    m.batch = batch;
    m.n_slots = c.page_table ? (int64_t)c.n_pages * H * c.page_tokens : (int64_t)batch * H * c.capacity;
    m.status = status;
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
    std::vector<uint8_t> in_bits;   // the plan's defining inputs, kept for bgtq_plan_save:
    std::vector<double> in_energy;  // block widths and energies [H][64]
    std::vector<uint32_t> img_src;  // decode table entries (see single_base)
    std::vector<uint32_t> cells;    // code-search cell tables (kCellHdr words, then the entries)
    int img_ws = 0;                 // widest code the decode tables cover
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
    int slack = 0;  // the newest range (split 0) holds about this many tokens fewer
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
