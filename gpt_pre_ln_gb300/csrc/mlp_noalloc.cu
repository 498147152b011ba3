// gpt2_mlp_noalloc: the MLP sublayer of gpt2_mlp without a caller-provided
// workspace, for callers that cannot allocate device memory when they call
// in.  Examples: a plug-in inside a serving process whose framework has
// already reserved the GPU's memory in its own pool and fails or mis-counts
// any allocation made behind its back; code that runs while a stream is
// being captured into a CUDA graph, where cudaMalloc is not permitted; and
// latency-critical paths that cannot afford cudaMalloc's implicit device
// synchronisation.
//
// The [M, F] hidden activation lives in a fixed scratch array in device
// global memory that this file owns (kMlpScratchBytes per GPU, held from the
// first use of the library on a device until the process exits).  Host code
// never uses the array's name as an address: the first call on each device
// looks up its device address with cudaGetSymbolAddress (with that device
// current) and caches it.  Nothing else is allocated, by this library or by
// any library it calls.
//
// The hidden activation is written completely by the c_fc GEMM before the
// MLP c_proj GEMM reads it, so no part of the array needs to start at zero.
// Every call on a device shares the one array: calls whose GPU work can
// overlap (different streams without ordering between them) race on it and
// produce wrong results; calls ordered on one stream are safe.
//
// The cached address belongs to the CUDA context it was looked up in.  A
// caller that resets a device (cudaDeviceReset) and keeps using the library
// in the same process gets a new context whose copy of the array may sit
// elsewhere; the cache is not refreshed, so such a caller must not use this
// entry point after the reset.
#include <climits>
#include <mutex>

#include "common.cuh"
#include "internal.h"

namespace gpt2 {
namespace {

constexpr size_t kMlpScratchBytes = size_t(16) << 20;  // 16 MiB per device

static __device__ __align__(256) unsigned char g_mlp_scratch[kMlpScratchBytes];

constexpr int kMaxDev = 64;
void* g_scratch_ptr[kMaxDev] = {nullptr};
std::mutex g_scratch_mu;

// Device address of the scratch array on the current device (nullptr if the
// lookup failed).  The first call per device does the lookup.
void* scratch_address() {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDev) return nullptr;
  std::lock_guard<std::mutex> lk(g_scratch_mu);
  if (!g_scratch_ptr[dev]) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_mlp_scratch) != cudaSuccess) return nullptr;
    g_scratch_ptr[dev] = p;
  }
  return g_scratch_ptr[dev];
}

inline bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

}  // namespace
}  // namespace gpt2

using namespace gpt2;

extern "C" {

size_t gpt2_mlp_noalloc_max_scratch_bytes(void) { return kMlpScratchBytes; }

int gpt2_mlp_noalloc(const void* x, const void* w_fc, const void* b_fc, const void* w_proj, const void* b_proj,
                     const float* residual, float* out, int64_t M, int D, int F, gpt2_dtype dtype,
                     gpt2_stream_t stream) {
  if (dtype != GPT2_F32 && dtype != GPT2_BF16 && dtype != GPT2_F16) return GPT2_ERR_ARG;
  if (M < 0 || M > INT_MAX || D <= 0 || F <= 0) return GPT2_ERR_ARG;
  if (D % 64 != 0 || F % 64 != 0) return GPT2_ERR_UNSUPPORTED;
  const size_t esz = dtype == GPT2_F32 ? 4 : 2;
  if (static_cast<size_t>(M) * static_cast<size_t>(F) * esz > kMlpScratchBytes) return GPT2_ERR_WORKSPACE;
  if (M == 0) return GPT2_OK;
  const void* ps[6] = {x, w_fc, b_fc, w_proj, b_proj, out};
  for (const void* p : ps)
    if (!p || !aligned16(p)) return GPT2_ERR_ARG;
  if (residual && !aligned16(residual)) return GPT2_ERR_ARG;
  void* g = scratch_address();
  if (!g) return GPT2_ERR_CUDA;
  // the same launches as gpt2_mlp, with the scratch array as the hidden buffer
  const cudaError_t e = launch_mlp(dtype, x, w_fc, b_fc, w_proj, b_proj, residual, out, M, D, F, g,
                                   reinterpret_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? GPT2_OK : GPT2_ERR_CUDA;
}

}  // extern "C"
