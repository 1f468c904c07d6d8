// Batched paged decode attention that allocates nothing.
//
// pkv_paged_decode_attention needs a caller-provided device workspace for the
// split kernel's partial results and the per-request tile prefix.  Some callers
// cannot obtain one: code embedded in a host application that has already
// reserved the GPU's memory for its own arena (a new cudaMalloc would fail or
// fragment it) and has no allocator to lend, or code on a latency-critical path
// that must not call cudaMalloc / cudaFree because those can synchronise the
// device and take milliseconds.  This entry point serves them: its scratch is a
// fixed array in this library's device memory, sized PKV_STATIC_SCRATCH_BYTES,
// which every GPU that loads the library holds until the process exits.
//
// The array is shared by every call on a device and keeps the previous call's
// contents.  Nothing in it needs to start at zero: the plan kernel writes the
// tile prefix and the worker table before any reader, and every partial slot the
// merge kernel reads is written by the split kernel of the same call.  Calls
// whose device work can overlap (different streams, or different host threads)
// race on the array; serialise them, e.g. on one stream.

#include <cuda_runtime.h>

#include <cstdint>

#include "pkv.h"
#include "pkv_internal.h"

namespace {

static __device__ __align__(256) unsigned char g_static_scratch[PKV_STATIC_SCRATCH_BYTES];

constexpr int kMaxDevices = 256;
// Device address of g_static_scratch per device, looked up once per device.
void* g_scratch_addr[kMaxDevices] = {};

}  // namespace

extern "C" int pkv_paged_decode_attention_static(pkv_pool* pool, int layer, int batch,
                                                 const float* q, const void* k_new,
                                                 const void* v_new, const int32_t* page_tables,
                                                 int max_pages, const int32_t* seq_lens,
                                                 int64_t max_seq_len, float* out, void* stream) {
    pkv::DecodeArgs a{};
    size_t need = 0;
    int rc = pkv::prepare_batched(pool, layer, batch, q, k_new, v_new, page_tables, max_pages,
                                  seq_lens, max_seq_len, out, &a, &need);
    if (rc != PKV_OK || a.B == 0) return rc;
    if (need > (size_t)PKV_STATIC_SCRATCH_BYTES)
        return pkv::record_error(
            PKV_ERR_INVALID_ARGUMENT,
            "batch %d x max_seq_len %lld needs %zu bytes of scratch, more than the %zu-byte "
            "static array; use pkv_paged_decode_attention with a workspace",
            batch, (long long)max_seq_len, need, (size_t)PKV_STATIC_SCRATCH_BYTES);
    int dev = -1;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess)
        return pkv::record_error(PKV_ERR_CUDA, "cudaGetDevice: %s", cudaGetErrorString(e));
    if (dev < 0 || dev >= kMaxDevices)
        return pkv::record_error(PKV_ERR_UNSUPPORTED, "device ordinal %d too large", dev);
    if (g_scratch_addr[dev] == nullptr) {
        // first call on this device (which is current): find the array's device address
        void* ptr = nullptr;
        e = cudaGetSymbolAddress(&ptr, g_static_scratch);
        if (e != cudaSuccess || ptr == nullptr)
            return pkv::record_error(PKV_ERR_CUDA, "cudaGetSymbolAddress of the static scratch: %s",
                                     cudaGetErrorString(e));
        g_scratch_addr[dev] = ptr;
    }
    a.workspace = g_scratch_addr[dev];
    a.workspace_bytes = PKV_STATIC_SCRATCH_BYTES;
    e = pkv::launch_decode(a, static_cast<cudaStream_t>(stream));
    if (e != cudaSuccess)
        return pkv::record_error(PKV_ERR_CUDA, "decode launch: %s", cudaGetErrorString(e));
    return pkv::record_error(PKV_OK, "");
}
