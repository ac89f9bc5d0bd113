// The parameter block and the prompt encoder shared by the prefill kernels
// (a whole prompt into an empty cache, a later chunk onto a cached prefix).
#pragma once

#include <cuda_fp16.h>

#include "encode.cuh"

namespace bgtq {
namespace {

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

// Encode the keys and values of cache positions [p0, p0 + n) of (b, h),
// read from rows p0 - shift .. of the given K/V (shift: the prefix length of
// a later chunk, 0 for a whole prompt): warp w takes the token pairs w,
// w + n_warps, ...; the steps are the append kernel's.  The fp16 recent-key
// ring (if any) receives the positions within p.recent of seq_end.
__device__ void encode_block(const PfParams& p, int b, int h, int p0, int n, int shift, int seq_end, const float* s_thr,
                             uint32_t (*s_rec)[8 * kPairMaxW], uint32_t* s_vmask, int warp, int lane, int n_warps) {
    const HeadTab* ht = p.heads + h;
    EncLane ek, ev;
    enc_lane_load(ek, ht, true, p.bv, p.v_inv_sqrt, lane);
    enc_lane_load(ev, ht, false, p.bv, p.v_inv_sqrt, lane);
    const size_t row0 = ((size_t)b * p.H + h) * p.T;
    const size_t unit = (size_t)b * p.H + h;
    for (int pi = warp; 2 * pi < n; pi += n_warps) {
        const int pos0 = p0 + 2 * pi;
        const bool has[2] = {true, 2 * pi + 1 < n};
        // ---- keys of the pair
        float x[2][4];
#pragma unroll
        for (int m = 0; m < 2; ++m) {
            const __half* row = p.k + (row0 + pos0 - shift + m) * kD;
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
            if (p.recent > 0 && pos >= seq_end - p.recent) {
                // fp16 recent-key ring: the key as given, slot pos mod W
                const uint2 nat = *(reinterpret_cast<const uint2*>(p.k + (row0 + pos - shift) * kD) + lane);
                *(reinterpret_cast<uint2*>(p.k_recent + (unit * p.recent + pos % p.recent) * kD) + lane) = nat;
            }
        }
        __syncwarp();
        // ---- values of the pair: one V record
#pragma unroll
        for (int m = 0; m < 2; ++m) {
            uint2 raw = make_uint2(0u, 0u);
            if (has[m]) raw = *(reinterpret_cast<const uint2*>(p.v + (row0 + pos0 - shift + m) * kD) + lane);
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

}  // namespace
}  // namespace bgtq
