// Bulk quantize-append kernels for 2-word K record slices (256 bits per key).
#include "codec_bulk.cuh"

namespace bgtq {

template <>
cudaError_t launch_bulk_bk<2>(const QParams& p, int bv, int batch, cudaStream_t s) {
    return launch_bulk_bk_impl<2>(p, bv, batch, s);
}

}  // namespace bgtq
