// Decode attention on the Block-GTQ packed cache: split planning, workspace
// sizes and launches of the contiguous-cache instances (the kernel is in
// decode_kernel.cuh; the paged-cache instances in decode_attn_paged.cu).
//
// Method: "RoPE-Aware Bit Allocation for KV-Cache Quantization" — English
// abstract and review §1 "Packed-Cache" / Figure 2: attention is computed on
// the compressed K/V, no fp16 KV cache is materialised.
#include <algorithm>
#include <cmath>
#include <map>
#include <mutex>
#include <tuple>

#include "decode_kernel.cuh"

namespace bgtq {
namespace {

// CTAs of decode_kernel<BK, BV> that can be resident at once, in whole
// clusters (cluster placement can leave SMs unusable, so this is at most
// the SM count times the blocks per SM).
template <int BK, int BV>
int resident_ctas(int ws) {
    if (ensure_smem_attr<BK, BV, false>() != cudaSuccess) {
        cudaGetLastError();
        return 0;
    }
    cudaLaunchAttribute attr[2];
    cudaLaunchConfig_t cfg = launch_config<BK, BV>(dim3(kCluster, 1, 1), nullptr, ws, attr);
    cfg.numAttrs = 1;  // occupancy: the cluster shape only
    int clusters = 0;
    if (cudaOccupancyMaxActiveClusters(&clusters, decode_kernel<BK, BV, 2, false>, &cfg) != cudaSuccess || clusters <= 0) {
        cudaGetLastError();
        return 0;
    }
    // never more than the SMs hold block by block (registers, shared memory)
    int per_sm = 0, dev = 0, sms = 0;
    cudaGetDevice(&dev);
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, decode_kernel<BK, BV, 2, false>, kWarps * 32,
                                                      cfg.dynamicSmemBytes) != cudaSuccess ||
        cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) {
        cudaGetLastError();
        return 0;
    }
    const int cap = per_sm * sms / kCluster * kCluster;
    return std::min(clusters * kCluster, cap);
}

int resident_ctas_for(int bk, int bv, int ws) {
    static std::mutex mu;
    static std::map<std::tuple<int, int, int>, int> cache;
    int dev = 0;
    cudaGetDevice(&dev);
    const int key = bk * 10 + bv;
    std::lock_guard<std::mutex> lock(mu);
    auto it = cache.find({dev, key, ws});
    if (it != cache.end()) return it->second;
    int n = 0;
    switch (key) {
        case 11: n = resident_ctas<1, 1>(ws); break;
        case 12: n = resident_ctas<1, 2>(ws); break;
        case 13: n = resident_ctas<1, 3>(ws); break;
        case 14: n = resident_ctas<1, 4>(ws); break;
        case 21: n = resident_ctas<2, 1>(ws); break;
        case 22: n = resident_ctas<2, 2>(ws); break;
        case 23: n = resident_ctas<2, 3>(ws); break;
        case 24: n = resident_ctas<2, 4>(ws); break;
        case 31: n = resident_ctas<3, 1>(ws); break;
        case 32: n = resident_ctas<3, 2>(ws); break;
        case 33: n = resident_ctas<3, 3>(ws); break;
        case 34: n = resident_ctas<3, 4>(ws); break;
        default: n = 0;
    }
    cache[{dev, key, ws}] = n;
    return n;
}

}  // namespace

SplitPlan decode_split(const bgtq_plan& p, int batch, int64_t max_len) {
    // One wave of resident CTAs in total (whole clusters), every split a
    // whole number of steps (kTile tokens for each warp of the CTA).
    constexpr int64_t kStepTok = kWarps * kTile;
    SplitPlan sp;
    const int64_t units = std::max<int64_t>(1, (int64_t)batch * p.H);
    const int64_t len = std::max<int64_t>(max_len, 1);
    int64_t slots = (p.bk >= 1 && p.bk <= 3 && p.bv >= 1 && p.bv <= 4)
                        ? resident_ctas_for(p.bk, p.bv, p.img_ws) : 0;
    if (slots <= 0) slots = std::max(1, p.num_sms);
    // Leave one cluster's room for a kernel that programmatic dependent
    // launch starts early next to this one, so that every cluster of this
    // grid can be resident at once.
    if (slots > 2 * kCluster) slots -= kCluster;
    int64_t ns = slots / units;
    if (ns >= kCluster) ns = ns / kCluster * kCluster;
    // Splits longer than kMaxSplitTokens are cut further (several waves):
    // in a ragged batch the long sequences then spread over many CTAs
    // instead of one CTA each, and the short sequences' extra splits exit
    // at once.
    ns = std::max<int64_t>(ns, (len + kMaxSplitTokens - 1) / kMaxSplitTokens);
    ns = std::min<int64_t>(ns, (len + kStepTok - 1) / kStepTok);
    ns = std::min<int64_t>(ns, (int64_t)kCluster * kMaxClusters);
    if (len >= kStepTok * kCluster) ns = std::max<int64_t>(ns, kCluster);
    ns = std::max<int64_t>(ns, 1);
    // The newest range (split 0) is shorter by `slack` tokens: in a fused
    // decode step its CTA first appends the new token (a few microseconds of
    // encoding).  The ranges are the same with and without the append, so
    // both paths merge identical partials.  Ranges are whole 16-token tiles.
    int64_t slack = 0, tps = 0;
    for (;; ++ns) {
        slack = std::min<int64_t>(256, (len + ns - 1) / ns / 4) / kTile * kTile;
        tps = (len + slack + ns - 1) / ns;
        tps = std::max<int64_t>((tps + kTile - 1) / kTile * kTile, kStepTok);
        if (tps <= kMaxSplitTokens) break;
        if (ns >= (int64_t)kCluster * kMaxClusters) {  // the longest sequences: no slack
            slack = 0;
            tps = std::max<int64_t>(((len + ns - 1) / ns + kTile - 1) / kTile * kTile, kStepTok);
            break;
        }
    }
    // splits the kernel makes active for a sequence of len tokens (at most
    // that for shorter ones): split 0 holds [a0, len), a0 = len - tps + slack
    // rounded up to a tile
    const int64_t a0 = std::max<int64_t>(0, (len - tps + slack + kTile - 1) / kTile * kTile);
    const int64_t n = 1 + (a0 + tps - 1) / tps;
    sp.tokens_per_split = (int)tps;
    sp.slack = (int)slack;
    sp.n_split = (int)((n + kCluster - 1) / kCluster * kCluster);
    return sp;
}

size_t decode_counter_bytes(const bgtq_plan& p, int batch) {
    return (((size_t)batch * p.H * p.G * sizeof(uint32_t)) + 255) / 256 * 256;
}

size_t decode_workspace_bytes(const bgtq_plan& p, int batch, const SplitPlan& sp) {
    const size_t units = (size_t)batch * p.H;
    const size_t counters = decode_counter_bytes(p, batch);
    return counters + units * (size_t)(sp.n_split / kCluster) * p.G * kPartStride * sizeof(float);
}

cudaError_t launch_decode(const bgtq_plan& pl, cudaStream_t s, const void* q, const bgtq_cache& c,
                          const int32_t* seq_lens, int batch, const SplitPlan& sp, void* out, int out_dtype,
                          float scale, void* ws, int32_t* status, const void* k_new, const void* v_new,
                          const int32_t* pos_new) {
    DecodeParams p;
    p.q = static_cast<const __half*>(q);
    p.kc = static_cast<uint8_t*>(c.k_codes);
    p.kn = c.k_norm;
    p.vc = static_cast<uint8_t*>(c.v_codes);
    p.vn = c.v_norm;
    p.cap = c.capacity;
    p.map = make_cache_map(c, pl.H, batch, status);
    p.seq_lens = seq_lens;
    p.out = out;
    p.out_dtype = out_dtype;
    const size_t counters = decode_counter_bytes(pl, batch);
    p.count = static_cast<uint32_t*>(ws);
    p.part = reinterpret_cast<float*>(static_cast<char*>(ws) + counters);
    p.heads = pl.dev.heads;
    p.img_src = pl.dev.img_src;
    p.img_lane = lane_entries(pl.img_ws);
    p.img_shared = shared_words(pl.img_ws);
    p.img_ws = pl.img_ws;
    p.img_bytes = 0;  // set at launch
    p.scale_log2 = scale * 1.4426950408889634f;
    p.v_inv_sqrt = (float)(1.0 / std::sqrt((double)kD));
    p.H = pl.H;
    p.G = pl.G;
    p.n_split = sp.n_split;
    p.tps = sp.tokens_per_split;
    p.slack = sp.slack;
    p.status = status;
    p.k_new = static_cast<const __half*>(k_new);
    p.v_new = static_cast<const __half*>(v_new);
    p.pos_new = pos_new;
    p.thr = pl.dev.thr;
    p.k_recent = static_cast<__half*>(c.k_recent);
    p.recent = c.recent;
    dim3 grid((unsigned)sp.n_split, (unsigned)pl.H, (unsigned)batch);
    // the fast instances decode codes of width >= 4 only in each lane's
    // kFastWide widest slots; the general instance in any slot, and it takes
    // a recent-key window longer than kWinPre
    bool any_wide = false;
    for (const HeadTab& ht : pl.heads) any_wide |= ht.n_wide > kFastWide;
    const int kind = any_wide ? 2 : (c.recent > 0 ? (c.recent <= kWinPre ? 1 : 2) : 0);
    if (c.page_table) return launch_decode_paged(p, grid, s, kind, pl.bk, pl.bv);
    const int key = pl.bk * 10 + pl.bv;
    switch (key) {
        case 11: return launch_t<1, 1, false>(p, grid, s, kind);
        case 12: return launch_t<1, 2, false>(p, grid, s, kind);
        case 13: return launch_t<1, 3, false>(p, grid, s, kind);
        case 14: return launch_t<1, 4, false>(p, grid, s, kind);
        case 21: return launch_t<2, 1, false>(p, grid, s, kind);
        case 22: return launch_t<2, 2, false>(p, grid, s, kind);
        case 23: return launch_t<2, 3, false>(p, grid, s, kind);
        case 24: return launch_t<2, 4, false>(p, grid, s, kind);
        case 31: return launch_t<3, 1, false>(p, grid, s, kind);
        case 32: return launch_t<3, 2, false>(p, grid, s, kind);
        case 33: return launch_t<3, 3, false>(p, grid, s, kind);
        case 34: return launch_t<3, 4, false>(p, grid, s, kind);
        default: return cudaErrorInvalidValue;
    }
}

}  // namespace bgtq
