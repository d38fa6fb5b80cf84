// cp_decode_attn_noalloc: the split-KV decode with its scratch in a fixed,
// library-owned device array instead of a caller-provided workspace.
//
// Who needs it: callers that cannot allocate device memory at the point of
// the call — real-time serving loops held to a fixed memory budget, and
// plugins reached through a C interface that gives them no allocator.  They
// pass inputs and outputs only; the partial results of KV ranges that the
// schedule splits across CTAs go to a static __device__ array.
//
// The array (CP_NOALLOC_SCRATCH_BYTES) is part of the library image: every
// GPU that loads the library holds it until the process exits.  Every call
// shares it and the array keeps the last call's contents.  No word of it has
// to start at zero: each scratch slot is written in full by the decode kernel
// before the merge kernel of the same call reads it.  Calls whose work
// overlaps on the GPU (different streams, or different host threads without
// ordering) race on the array and corrupt each other's results; serialise
// them on one stream.
//
// Host code cannot pass the symbol itself to a kernel (in host code it names a
// host-side stand-in).  The device address comes from cudaGetSymbolAddress
// with the query's device current.  It is looked up again on every call made
// while the stream is not capturing (so a context torn down and re-created,
// e.g. after cudaDeviceReset, never leaves a stale address behind); a call on
// a capturing stream uses the address cached by the last such lookup on that
// device, so the first call on a device must come before any stream capture.
#include <mutex>

#include "internal.h"

namespace {

static __device__ __align__(256) unsigned char g_noalloc_scratch[CP_NOALLOC_SCRATCH_BYTES];

std::mutex g_scratch_mu;
void* g_scratch_ptr[256] = {nullptr};

cudaError_t scratch_address(int dev, cudaStream_t stream, void** out) {
  if (dev < 0 || dev >= 256) return cudaErrorInvalidDevice;
  cudaStreamCaptureStatus cap = cudaStreamCaptureStatusNone;
  cudaError_t e = cudaStreamIsCapturing(stream, &cap);
  if (e != cudaSuccess) return e;
  std::lock_guard<std::mutex> lock(g_scratch_mu);
  if (cap == cudaStreamCaptureStatusNone) {
    void* p = nullptr;
    e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
    if (e != cudaSuccess) return e;
    if (!p) return cudaErrorInvalidSymbol;
    g_scratch_ptr[dev] = p;
  } else if (!g_scratch_ptr[dev]) {
    return cudaErrorStreamCaptureUnsupported;  // no earlier call on this device
  }
  *out = g_scratch_ptr[dev];
  return cudaSuccess;
}

}  // namespace

extern "C" cp_status cp_decode_attn_noalloc(const void* host_plan, const void* dev_plan,
                                            cp_decode_mode mode, cp_dtype kv_dtype, const void* q,
                                            const void* const* shard_k,
                                            const void* const* shard_v,
                                            const float* const* shard_scale, int Hq, int Hkv,
                                            int Dqk, int Dv, float sm_scale, float* o_part,
                                            float* lse_part, void* stream) {
  size_t need = 0;
  cp_status st = cp_decode_workspace_size(host_plan, Hq, Dv, &need);
  if (st != CP_OK) return st;
  if (need > (size_t)CP_NOALLOC_SCRATCH_BYTES)
    return cpattn::report_error(
        CP_ERR_WORKSPACE,
        "cp_decode_attn_noalloc: this plan needs %zu bytes of scratch, more than the fixed "
        "%zu-byte array; call cp_decode_attn with a workspace, or plan with fewer workers",
        need, (size_t)CP_NOALLOC_SCRATCH_BYTES);
  // The array used is the current device's: q must live on that device.
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess)
    return cpattn::report_error(CP_ERR_CUDA, "cp_decode_attn_noalloc: cudaGetDevice failed: %s",
                                cudaGetErrorString(e));
  if (q) {
    cudaPointerAttributes attr;
    e = cudaPointerGetAttributes(&attr, q);
    if (e != cudaSuccess) {
      cudaGetLastError();
      return cpattn::report_error(CP_ERR_INVALID_ARG,
                                  "cp_decode_attn_noalloc: q is not a device pointer");
    }
    if (attr.type == cudaMemoryTypeDevice && attr.device != dev)
      return cpattn::report_error(
          CP_ERR_INVALID_ARG,
          "cp_decode_attn_noalloc: q lives on device %d but device %d is current; make q's "
          "device current before the call",
          attr.device, dev);
  }
  void* scratch = nullptr;
  e = scratch_address(dev, static_cast<cudaStream_t>(stream), &scratch);
  if (e != cudaSuccess)
    return cpattn::report_error(CP_ERR_CUDA,
                                "cp_decode_attn_noalloc: looking up the scratch array failed "
                                "(the first call on a device must not be on a capturing "
                                "stream): %s",
                                cudaGetErrorString(e));
  return cp_decode_attn(host_plan, dev_plan, mode, kv_dtype, q, shard_k, shard_v, shard_scale, Hq,
                        Hkv, Dqk, Dv, sm_scale, o_part, lse_part, scratch,
                        (size_t)CP_NOALLOC_SCRATCH_BYTES, stream);
}

extern "C" size_t cp_noalloc_scratch_bytes(void) { return (size_t)CP_NOALLOC_SCRATCH_BYTES; }
