// TQ-MSE encoder (quantize-append) and decoder (debug dequant) for the
// Block-GTQ packed cache.
//
// Method: "RoPE-Aware Bit Allocation for KV-Cache Quantization" — review §1
// Key Terms (TQ-MSE rotates then quantises; the packed cache stores
// compressed K/V) and English abstract (per-block integer widths for keys,
// uniform TQ-MSE for values).  A warp encodes tokens two at a time: lane L
// holds codec coordinates 4L..4L+3 of each.  Every float operation is a single correctly rounded
// IEEE operation in a fixed order (this file is built with --fmad=false and
// uses explicit _rn intrinsics), so codes, norms and decoded values are
// bit-identical to any implementation that follows the same steps.
#include <cuda_fp16.h>

#include "bgtq_internal.h"
#include "encode.cuh"

namespace bgtq {
namespace {

constexpr int kWarpsQ = 4;
constexpr int kPairsPerBlock = 16;  // token pairs each quantize_append block encodes


// One block appends up to kPairsPerBlock token pairs of one (sequence, head).
// Warps 0 and 1 encode keys (the even and the odd token of each pair, two
// pairs at a time), warps 2 and 3 encode values (alternate pairs, both tokens
// of a pair at once, since a V record holds a token pair).  Each warp loads
// the rows of its next group before encoding the current one.  A pair that
// is only half appended has its V record merged in place with atomic AND/OR,
// so nothing is read back.
__global__ void __launch_bounds__(128) quantize_append_kernel(QParams p) {
    __shared__ float s_thr[kThrCompact];
    __shared__ uint32_t rec[kWarpsQ][2][8 * kPairMaxW];  // records being assembled per warp
    __shared__ uint32_t rmask[2][8 * kPairMaxW];
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int h = blockIdx.y, b = blockIdx.z;
    // The next kernel may launch right away (programmatic dependent launch).
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");

    // ---- plan-static set-up, before waiting for the previous kernel
    stage_thresholds(s_thr, p.thr, threadIdx.x, kWarpsQ * 32);
    const HeadTab* ht = p.heads + h;
    const size_t unit = (size_t)b * p.H + h;
    const bool is_k = warp < 2;
    EncLane el;
    enc_lane_load(el, ht, is_k, p.bv, p.v_inv_sqrt, lane);
    __syncthreads();
    // pos_start is read before the wait: no kernel of this library writes it
    const int ps = p.pos_start[b];
    asm volatile("griddepcontrol.wait;" ::: "memory");
    if (ps < 0 || (int64_t)ps + p.t_new > p.cap) {
        if (blockIdx.x == 0 && h == 0 && threadIdx.x == 0 && p.status) {
            atomicOr(p.status, BGTQ_STATUS_APPEND_CAPACITY);
            debug_in_range(false, p.status);  // positions past the capacity
        }
        return;
    }
    const int64_t end = (int64_t)ps + p.t_new;
    const int64_t P0 = (int64_t)(ps >> 1) + (int64_t)blockIdx.x * kPairsPerBlock;

    if (is_k) {
        // ---- keys: warp w encodes tokens 2P + w of pairs P = P0 + i, i + 1
        const int krec_words = 4 * p.bk;
        auto load = [&](int i, __half (&xh)[2][4]) {
#pragma unroll
            for (int n = 0; n < 2; ++n) {
                const int64_t pos = 2 * (P0 + i + n) + warp;
                if (pos >= ps && pos < end) {
                    const __half* row = p.k + (unit * p.t_new + (size_t)(pos - ps)) * kD;
#pragma unroll
                    for (int k = 0; k < 4; ++k) xh[n][k] = row[el.src[k]];
                }
            }
        };
        __half cur[2][4], nxt[2][4];
        load(0, cur);
        for (int i = 0; i < kPairsPerBlock; i += 2) {
            if (2 * (P0 + i) + warp >= end) break;
            if (i + 2 < kPairsPerBlock) load(i + 2, nxt);
            bool has[2];
            float x[2][4];
#pragma unroll
            for (int n = 0; n < 2; ++n) {
                const int64_t pos = 2 * (P0 + i + n) + warp;
                has[n] = pos >= ps && pos < end;
#pragma unroll
                for (int k = 0; k < 4; ++k) x[n][k] = has[n] ? __fmul_rn(__half2float(cur[n][k]), el.wh[k]) : 0.0f;
            }
            int code[2][4];
            float rho[2];
            for (int k = lane; k < 2 * 8 * kPairMaxW; k += 32) (&rec[warp][0][0])[k] = 0;
            __syncwarp();
            warp_encode_n<2>(x, el.sg, el.pl, el.is, el.wd, el.n_coded, s_thr, code, rho);
#pragma unroll
            for (int n = 0; n < 2; ++n) pack_k_fields(rec[warp][n], code[n], el, lane);
            __syncwarp();
#pragma unroll
            for (int n = 0; n < 2; ++n) {
                if (!has[n]) continue;
                const int64_t pos = 2 * (P0 + i + n) + warp;
                const int64_t sl = p.map.slot(b, h, pos);
                if (sl < 0) {
                    if (lane == 0 && p.status) atomicOr(p.status, BGTQ_STATUS_PAGE_RANGE);
                    continue;
                }
                uint32_t* dst = reinterpret_cast<uint32_t*>(p.kc + sl * (16 * p.bk));
                if (lane < krec_words) dst[lane] = rec[warp][n][lane];
                if (lane == 0) p.kn[sl] = rho[n];
                if (p.recent > 0 && pos >= end - p.recent) {
                    // fp16 recent-key ring: the key as given, slot pos mod W
                    const uint2 nat = *(reinterpret_cast<const uint2*>(p.k + (unit * p.t_new + (size_t)(pos - ps)) * kD) + lane);
                    *(reinterpret_cast<uint2*>(p.k_recent + (unit * p.recent + pos % p.recent) * kD) + lane) = nat;
                }
            }
            __syncwarp();
#pragma unroll
            for (int n = 0; n < 2; ++n)
#pragma unroll
                for (int k = 0; k < 4; ++k) cur[n][k] = nxt[n][k];
        }
        return;
    }

    // ---- values: warp 2 + r encodes both tokens of pairs P0 + r, P0 + r + 2, ...
    const int r = warp - 2;
    const int vrec_words = 8 * p.bv;
    uint32_t* vrec = rec[warp][0];
    uint32_t* vmask = rmask[r];
    auto load = [&](int i, uint2 (&xr)[2]) {
        const int64_t pos0 = 2 * (P0 + i);
#pragma unroll
        for (int par = 0; par < 2; ++par) {
            const int64_t pos = pos0 + par;
            if (pos >= ps && pos < end)
                xr[par] = *(reinterpret_cast<const uint2*>(p.v + (unit * p.t_new + (size_t)(pos - ps)) * kD) + lane);
        }
    };
    uint2 cur[2] = {make_uint2(0, 0), make_uint2(0, 0)}, nxt[2] = {make_uint2(0, 0), make_uint2(0, 0)};
    load(r, cur);
    for (int i = r; i < kPairsPerBlock; i += 2) {
        const int64_t P = P0 + i;
        const int64_t pos0 = 2 * P;
        if (pos0 >= end) break;
        if (i + 2 < kPairsPerBlock) load(i + 2, nxt);
        const bool has[2] = {pos0 >= ps, pos0 + 1 < end};
        float x[2][4];
#pragma unroll
        for (int par = 0; par < 2; ++par) {
            const float2 a = __half22float2(*reinterpret_cast<const __half2*>(&cur[par].x));
            const float2 c = __half22float2(*reinterpret_cast<const __half2*>(&cur[par].y));
            x[par][0] = has[par] ? a.x : 0.0f;
            x[par][1] = has[par] ? a.y : 0.0f;
            x[par][2] = has[par] ? c.x : 0.0f;
            x[par][3] = has[par] ? c.y : 0.0f;
        }
        for (int k = lane; k < 8 * kPairMaxW; k += 32) {
            vrec[k] = 0;
            vmask[k] = 0;
        }
        __syncwarp();
        int code[2][4];
        float rho[2];
        warp_encode_n<2>(x, el.sg, el.pl, el.is, el.wd, kD, s_thr, code, rho);
        const int64_t sl0 = p.map.slot(b, h, pos0);  // the pair's page (pos0 even)
        if (sl0 < 0 && lane == 0 && p.status) atomicOr(p.status, BGTQ_STATUS_PAGE_RANGE);
#pragma unroll
        for (int par = 0; par < 2; ++par) {
            if (!has[par]) continue;
            pack_v_fields(vrec, vmask, code[par], par, p.bv, lane);
            if (lane == 0 && sl0 >= 0) p.vn[sl0 + par] = rho[par];
        }
        __syncwarp();
        uint32_t* vdst = reinterpret_cast<uint32_t*>(p.vc + (sl0 >> 1) * (32 * p.bv));
        for (int k = lane; k < vrec_words && sl0 >= 0; k += 32) {
            if (has[0] && has[1]) {
                vdst[k] = vrec[k];
            } else {
                // merge the appended half into the record without reading it
                atomicAnd(vdst + k, ~vmask[k]);
                atomicOr(vdst + k, vrec[k]);
            }
        }
        __syncwarp();
        cur[0] = nxt[0];
        cur[1] = nxt[1];
    }
}

struct DqParams {
    const uint8_t* kc;
    const float* kn;
    const uint8_t* vc;
    const float* vn;
    int64_t cap, t0, t1;
    CacheMap map;
    int b, h;
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
    int64_t sl = p.map.slot(p.b, p.h, t);
    if (sl < 0) sl = 0;  // page index out of range: unspecified output
    if (p.k_out) {
        const uint32_t* src = reinterpret_cast<const uint32_t*>(p.kc + sl * (16 * p.bk));
        if (lane < 4 * p.bk) rec[warp][lane] = src[lane];
        __syncwarp();
        const float rho = p.kn[sl];
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
                y[i] = debug_in_range(w <= kWMax && c < (1u << w), nullptr) ? __fmul_rn(rho, p.cent[256 * w + c]) : 0.0f;
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
        const uint32_t* src = reinterpret_cast<const uint32_t*>(p.vc + (sl >> 1) * (32 * p.bv));
        for (int i = lane; i < 8 * p.bv; i += 32) rec[warp][i] = src[i];
        __syncwarp();
        const float rho = p.vn[sl];
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
            y[i] = debug_in_range(p.bv <= kWMax && c < (1u << p.bv), nullptr) ? __fmul_rn(rho, p.cent[256 * p.bv + c]) : 0.0f;
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
    p.map = make_cache_map(c, pl.H, batch, status);
    p.heads = pl.dev.heads;
    p.thr = pl.dev.thr;
    p.cells = pl.dev.cells;
    p.cell_words = (int)pl.cells.size();
    p.bk = pl.bk;
    p.bv = pl.bv;
    p.v_inv_sqrt = (float)(1.0 / std::sqrt((double)kD));
    p.status = status;
    p.k_recent = static_cast<__half*>(c.k_recent);
    p.recent = c.recent;
    cudaLaunchConfig_t cfg = {};
    cfg.stream = s;
    cudaLaunchAttribute attr;
    attr.id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr.val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = &attr;
    cfg.numAttrs = 1;
    // Bulk appends (prefill) take the two-lanes-per-token kernel, which reads
    // whole fp16 rows with 16-byte loads (its grid's z holds two blocks per
    // sequence); small appends (decode), other widths and batches of more
    // than 32767 sequences the warp-per-token kernel.
    const bool aligned = ((reinterpret_cast<uintptr_t>(k) | reinterpret_cast<uintptr_t>(v)) & 15) == 0;
    if (t_new >= kBulkMinTokens && aligned && pl.bk >= 1 && pl.bk <= 3 && pl.bv >= 1 && pl.bv <= 4 && batch <= 32767)
        return launch_quantize_append_bulk(p, pl.bk, pl.bv, batch, s);
    const int64_t pairs = (int64_t)t_new / 2 + 1;
    const int64_t per_block = kPairsPerBlock;
    cfg.gridDim = dim3((unsigned)((pairs + per_block - 1) / per_block), (unsigned)pl.H, (unsigned)batch);
    cfg.blockDim = dim3(32 * kWarpsQ, 1, 1);
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
    p.map = make_cache_map(c, pl.H, batch, nullptr);
    p.b = b;
    p.h = head;
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
