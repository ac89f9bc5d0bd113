// bgtq_decode_attn_noalloc: decode attention whose split-merge scratch lives
// in a fixed device array of this library instead of a caller workspace.
//
// Some callers cannot allocate device memory at the point where they run
// decode attention: code that runs under a custom allocator or memory pool
// that must not be bypassed, runtimes that forbid cudaMalloc after start-up
// (fixed memory budgets, some inference servers and plugin hosts), or callers
// that simply have no device-memory API of their own.  This entry point needs
// no workspace argument: every call uses one file-scope device array of
// kScratchBytes bytes, which every GPU that loads the library keeps until the
// process exits.
//
// Rules for callers:
//   - Every call looks up the array's device address on the current device
//     (cudaGetSymbolAddress, a host-side lookup, not a stream operation), so
//     a context that was reset and re-created gets the array's new address.
//     The first call on a device may load the library's device code into the
//     context; make that first call before any stream capture.
//   - All calls share the array and it keeps the last call's contents, so
//     calls that overlap on the GPU (different streams, no ordering) race and
//     give wrong results.  Calls ordered on one stream are fine.
//   - Problems whose merge scratch would exceed kScratchBytes are rejected
//     with BGTQ_ERR_WORKSPACE; use bgtq_decode_attn with a workspace instead.
#include <cmath>

#include "bgtq_internal.h"

namespace bgtq {
namespace {

constexpr size_t kScratchBytes = (size_t)2 << 20;  // 2 MiB
static __device__ __align__(256) unsigned char g_decode_scratch[kScratchBytes];

// Device address of g_decode_scratch in the current device's context.  Looked
// up on every call rather than cached per device ordinal: after
// cudaDeviceReset (or a released primary context) the module is loaded again
// and the array may live at another address.
int scratch_address(void** out) {
    int dev = -1;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return set_error(BGTQ_ERR_CUDA, "cudaGetDevice: %s", cudaGetErrorString(e));
    void* ptr = nullptr;
    e = cudaGetSymbolAddress(&ptr, g_decode_scratch);
    if (e != cudaSuccess || !ptr)
        return set_error(BGTQ_ERR_CUDA, "cudaGetSymbolAddress(decode scratch) on device %d: %s", dev,
                         cudaGetErrorString(e));
    *out = ptr;
    return BGTQ_OK;
}

}  // namespace
}  // namespace bgtq

using namespace bgtq;

extern "C" int bgtq_decode_attn_noalloc(const bgtq_plan* p, void* stream, const void* q, const bgtq_cache* c,
                                        const int32_t* seq_lens, int64_t max_len, int batch, void* out,
                                        int out_dtype, float scale, int32_t* status) {
    if (!p) return set_error(BGTQ_ERR_INVALID_ARG, "plan is NULL");
    if (p->flags & BGTQ_PLAN_HOST_ONLY) return set_error(BGTQ_ERR_INVALID_ARG, "plan was built host-only");
    if (int rc = check_cache(p, c)) return rc;
    if (batch < 0 || max_len < 0) return set_error(BGTQ_ERR_INVALID_ARG, "batch and max_len must be >= 0");
    if (batch == 0) return BGTQ_OK;
    if (!q || !seq_lens || !out) return set_error(BGTQ_ERR_INVALID_ARG, "NULL pointer");
    if (out_dtype != 0 && out_dtype != 1) return set_error(BGTQ_ERR_INVALID_ARG, "out_dtype must be 0 (half) or 1 (float)");
    if (p->bk > 3) return set_error(BGTQ_ERR_UNSUPPORTED, "decode supports bits_per_key <= 384");
    if (p->bv > 4) return set_error(BGTQ_ERR_UNSUPPORTED, "decode supports v_bits <= 4");
    if (!(scale > 0.0f) || !std::isfinite(scale)) return set_error(BGTQ_ERR_INVALID_ARG, "softmax_scale must be finite and > 0");
    if (max_len > c->capacity) max_len = c->capacity;
    const SplitPlan sp = decode_split(*p, batch, max_len);
    const size_t need = decode_workspace_bytes(*p, batch, sp);
    if (need > kScratchBytes)
        return set_error(BGTQ_ERR_WORKSPACE,
                         "this problem needs %zu bytes of merge scratch; the built-in scratch holds %zu "
                         "(use bgtq_decode_attn with a workspace)", need, kScratchBytes);
    void* scratch = nullptr;
    int rc = scratch_address(&scratch);
    if (rc) return rc;
    // the arrival counters at the front must start at zero
    const size_t counter_bytes = decode_counter_bytes(*p, batch);
    cudaError_t e = cudaMemsetAsync(scratch, 0, counter_bytes, (cudaStream_t)stream);
    if (e != cudaSuccess) return set_error(BGTQ_ERR_CUDA, "clearing scratch counters: %s", cudaGetErrorString(e));
    e = launch_decode(*p, (cudaStream_t)stream, q, *c, seq_lens, batch, sp, out, out_dtype, scale, scratch, status);
    if (e != cudaSuccess) return set_error(BGTQ_ERR_CUDA, "decode_attn launch: %s", cudaGetErrorString(e));
    return BGTQ_OK;
}
