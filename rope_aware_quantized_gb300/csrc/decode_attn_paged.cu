// Decode attention on a paged Block-GTQ cache (pools of P-token pages and a
// page table per sequence): the paged instances of the decode kernel.  The
// kernel, shared with contiguous caches, is in decode_kernel.cuh; only the
// staging addresses, the L2 prefetch and the fused append's record location
// differ (a 16-token tile never straddles a page).
#include "decode_kernel.cuh"

namespace bgtq {

cudaError_t launch_decode_paged(const DecodeParams& p, dim3 grid, cudaStream_t s, int kind, int bk, int bv) {
    switch (bk * 10 + bv) {
        case 11: return launch_t<1, 1, true>(p, grid, s, kind);
        case 12: return launch_t<1, 2, true>(p, grid, s, kind);
        case 13: return launch_t<1, 3, true>(p, grid, s, kind);
        case 14: return launch_t<1, 4, true>(p, grid, s, kind);
        case 21: return launch_t<2, 1, true>(p, grid, s, kind);
        case 22: return launch_t<2, 2, true>(p, grid, s, kind);
        case 23: return launch_t<2, 3, true>(p, grid, s, kind);
        case 24: return launch_t<2, 4, true>(p, grid, s, kind);
        case 31: return launch_t<3, 1, true>(p, grid, s, kind);
        case 32: return launch_t<3, 2, true>(p, grid, s, kind);
        case 33: return launch_t<3, 3, true>(p, grid, s, kind);
        case 34: return launch_t<3, 4, true>(p, grid, s, kind);
        default: return cudaErrorInvalidValue;
    }
}

}  // namespace bgtq
