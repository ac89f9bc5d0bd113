// Bulk quantize-append kernels for 3-word K record slices (384 bits per key).
#include "codec_bulk.cuh"

namespace bgtq {

template <>
cudaError_t launch_bulk_bk<3>(const QParams& p, int bv, int batch, cudaStream_t s) {
    return launch_bulk_bk_impl<3>(p, bv, batch, s);
}

cudaError_t launch_quantize_append_bulk(const QParams& p, int bk, int bv, int batch, cudaStream_t s) {
    switch (bk) {
        case 1: return launch_bulk_bk<1>(p, bv, batch, s);
        case 2: return launch_bulk_bk<2>(p, bv, batch, s);
        case 3: return launch_bulk_bk<3>(p, bv, batch, s);
        default: return cudaErrorInvalidValue;
    }
}

}  // namespace bgtq
