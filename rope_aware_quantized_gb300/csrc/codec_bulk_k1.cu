// Bulk quantize-append kernels for 1-word K record slices (128 bits per key).
#include "codec_bulk.cuh"

namespace bgtq {

template <>
cudaError_t launch_bulk_bk<1>(const QParams& p, int bv, int batch, cudaStream_t s) {
    return launch_bulk_bk_impl<1>(p, bv, batch, s);
}

}  // namespace bgtq
