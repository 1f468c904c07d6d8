// Batched paged decode attention that allocates nothing.
//
// pkv_paged_decode_attention needs a caller-provided device workspace for the
// split kernel's partial results and the per-request tile prefix.  Some callers
// cannot obtain one: code embedded in a host application that has already
// reserved the GPU's memory for its own arena (a new cudaMalloc would fail or
// fragment it) and has no allocator to lend, or code on a latency-critical path
// that must not call cudaMalloc / cudaFree because those can synchronise the
// device and take milliseconds.  This entry point serves them: its scratch is a
// fixed array in this library's device memory, sized PKV_STATIC_SCRATCH_BYTES.
//
// When the array comes into being.  This file holds no kernel, so it is a module
// of its own, and under the CUDA runtime's lazy module loading (the default) the
// module -- and with it the array's 8 MiB -- is loaded in a context only when
// something first asks for the array's address.  pkv_pool_create does that, on
// the pool's device (static_scratch_address below), so the array is in place
// before the caller's decode loop and before an application reserves the rest of
// the GPU's memory; from then on it stays until the context is destroyed.
//
// The array is shared by every call on a device and keeps the previous call's
// contents.  What must start at zero is cleared on every call: the per-lane
// arrival counters at the start of the scratch, which the last arriving worker
// of a lane relies on, are zeroed by the plan kernel of each batched call (a
// batched call always runs its plan kernel; epoch-tagged counters are used only
// by the single-request path, which never comes here).  The plan kernel also
// writes the tile prefix and the worker table before any reader, and every
// partial slot the merge reads is written by the split kernel of the same call.
// Calls whose device work can overlap (different streams, or different host
// threads) race on the array; serialise them, e.g. on one stream.

#include <cuda_runtime.h>

#include <cstdint>

#include "pkv.h"
#include "pkv_internal.h"

namespace {

static __device__ __align__(256) unsigned char g_static_scratch[PKV_STATIC_SCRATCH_BYTES];

}  // namespace

namespace pkv {

// Device address of the array in the current context.  The name g_static_scratch
// in host code is a host-side stand-in, not a device address; this asks the
// runtime for the real one.  The first request in a context loads this file's
// module (and so the array); later ones are a lookup.  Not cached: after a
// device reset, or in another context of the same device, the address differs.
cudaError_t static_scratch_address(void** ptr) {
    *ptr = nullptr;
    return cudaGetSymbolAddress(ptr, g_static_scratch);
}

}  // namespace pkv

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
    // the lane counters in the array are zeroed by this call's plan kernel only
    if (a.epoch != 0)
        return pkv::record_error(PKV_ERR_BAD_STATE, "batched call with epoch-tagged counters");
    void* ptr = nullptr;
    cudaError_t e = pkv::static_scratch_address(&ptr);
    if (e != cudaSuccess || ptr == nullptr)
        return pkv::record_error(PKV_ERR_CUDA, "cudaGetSymbolAddress of the static scratch: %s",
                                 cudaGetErrorString(e));
    a.workspace = ptr;
    a.workspace_bytes = PKV_STATIC_SCRATCH_BYTES;
    e = pkv::launch_decode(a, static_cast<cudaStream_t>(stream));
    if (e != cudaSuccess)
        return pkv::record_error(PKV_ERR_CUDA, "decode launch: %s", cudaGetErrorString(e));
    return pkv::record_error(PKV_OK, "");
}
