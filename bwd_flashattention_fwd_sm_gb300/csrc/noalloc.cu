// Backward pass for callers that cannot allocate device memory.
//
// Some callers may not call cudaMalloc at all: engines that fix their device
// memory budget at start-up and forbid any allocation afterwards, and plug-ins
// living inside a host framework that owns the device allocator and shares none
// of it.  They cannot hand the library a workspace.  attn_bwd_noalloc serves
// them: its scratch space is a fixed array in this library's own device memory,
// created when the library's device code is loaded on a GPU and held until the
// process exits.
//
// The array is shared by every call: calls whose work overlaps on the GPU race on
// it (queue them on one stream, or wait between them).  Nothing in it has to
// survive from one call to the next: the backward rebuilds its work list and
// transposed mask, and its preprocess kernel zeroes the dQ accumulator every
// call before any kernel adds into it.
#include <cstdio>
#include <mutex>

#include "../../include/gbattn.h"
#include "common.cuh"

namespace gbattn {
void set_last_error_text(const char* text);
}

namespace {

static __device__ __align__(256) unsigned char g_noalloc_scratch[ATTN_NOALLOC_SCRATCH_BYTES];

constexpr int kMaxDevices = 64;
std::mutex g_mutex;
void* g_scratch_addr[kMaxDevices] = {nullptr};

}  // namespace

extern "C" attn_status_t attn_bwd_noalloc(const attn_params_t* p, const void* q, const void* k, const void* v,
                                          const void* o, const void* dout, const float* lse, void* dq, void* dk,
                                          void* dv, void* stream) {
  const size_t need = attn_bwd_workspace_size(p);
  // Invalid parameters: attn_bwd repeats the validation and returns its exact
  // code before touching anything.
  if (need == SIZE_MAX) return attn_bwd(p, q, k, v, o, dout, lse, dq, dk, dv, nullptr, 0, stream);
  if (need > ATTN_NOALLOC_SCRATCH_BYTES) {
    // attn_bwd's own pointer checks come first, so a bad pointer gets the same
    // code here as there; with no workspace it stops at its workspace check,
    // before anything is queued.
    const attn_status_t s = attn_bwd(p, q, k, v, o, dout, lse, dq, dk, dv, nullptr, 0, stream);
    if (s != ATTN_ERR_WORKSPACE) return s;
    char buf[200];
    snprintf(buf, sizeof(buf),
             "attn_bwd_noalloc: this problem needs %zu bytes of scratch, above the fixed %zu-byte array; "
             "use attn_bwd with a caller-provided workspace",
             need, (size_t)ATTN_NOALLOC_SCRATCH_BYTES);
    gbattn::set_last_error_text(buf);
    return ATTN_ERR_WORKSPACE;
  }
  void* scratch = nullptr;
  if (need > 0) {
    // In host code the array's name is only a stand-in; its device address is
    // looked up once per device, with that device current.
    int dev = -1;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess || dev < 0 || dev >= kMaxDevices) {
      gbattn::set_last_error_text("attn_bwd_noalloc: no usable CUDA device");
      return ATTN_ERR_CUDA;
    }
    std::lock_guard<std::mutex> lock(g_mutex);
    if (!g_scratch_addr[dev]) {
      void* ptr = nullptr;
      e = cudaGetSymbolAddress(&ptr, g_noalloc_scratch);
      if (e != cudaSuccess || !ptr) {
        char buf[160];
        snprintf(buf, sizeof(buf), "attn_bwd_noalloc: scratch address lookup failed: %s", cudaGetErrorString(e));
        gbattn::set_last_error_text(buf);
        return ATTN_ERR_CUDA;
      }
      g_scratch_addr[dev] = ptr;
    }
    scratch = g_scratch_addr[dev];
  }
  return attn_bwd(p, q, k, v, o, dout, lse, dq, dk, dv, scratch, ATTN_NOALLOC_SCRATCH_BYTES, stream);
}
