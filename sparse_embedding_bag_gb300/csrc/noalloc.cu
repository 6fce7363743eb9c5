// Allocation-free entry point: the unpooled atomic SGD update without a plan.
//
// Some callers cannot allocate device memory at the point where they run the
// backward pass: code that runs inside a CUDA graph capture (where cudaMalloc
// is not allowed), runtimes that hand out all device memory up front from
// their own pools, or embedders that forbid the library from touching the
// device allocator. Every other entry point needs a plan, and creating a plan
// calls cudaMalloc for its scratch. This one needs no plan: its scratch (the
// per-call control block, the error word and the 32-bit table offsets, about
// 21 KB) is the file-scope array below, which is part of the
// library's device image: it exists on every GPU that loads the library and
// stays there until the process exits. Its size bounds the problem:
// at most kNoAllocMaxN lookups and kMaxT tables per call.
//
// All calls (on every stream) share that one array and it keeps the last
// call's contents; the parts that must start at zero are cleared at the start
// of each call. Calls that overlap on the GPU race on it, so callers must
// order them (one stream, or events).
#include <cstddef>
#include <mutex>

#include "../../include/embbwd.h"
#include "decode.cuh"
#include "internal.cuh"

namespace embbwd {
namespace {

constexpr int64_t kNoAllocMaxN = (int64_t)1 << 22;  // lookups per call
constexpr int kNoAllocMaxDevices = 64;

struct NoAllocScratch {
  Ctl ctl;              // zeroed each call
  uint32_t status;      // zeroed each call; error bits of this call
  uint32_t pad[63];
  uint32_t hsc[kMaxT + 1];
};

static __device__ __align__(256) unsigned char g_noalloc_scratch[sizeof(NoAllocScratch)];

std::mutex g_mu;
void* g_addr[kNoAllocMaxDevices] = {};

// Set-up, once per device with that device current: the device address of the
// scratch array, and the shared-memory limits of the kernels it launches.
cudaError_t scratch_address(int device, NoAllocScratch** out) {
  std::lock_guard<std::mutex> lock(g_mu);
  if (!g_addr[device]) {
    void* ptr = nullptr;
    cudaError_t e = cudaGetSymbolAddress(&ptr, g_noalloc_scratch);
    if (e != cudaSuccess) return e;
    e = sort_configure(DevProps{0, 0});
    if (e != cudaSuccess) return e;
    g_addr[device] = ptr;
  }
  *out = static_cast<NoAllocScratch*>(g_addr[device]);
  return cudaSuccess;
}

// hash_size_cumsum (int64, device) -> 32-bit copy in the scratch, with the
// checks emb_bwd_plan does on the host: hash_size_cumsum starts at 0, is
// strictly increasing and < 2^32; every weights_offsets[t] is >= 0 and a
// multiple of 4 (the atomic scatter adds 16-byte vectors at
// weights + weights_offsets[t] + idx * D). A failed check sets kErrOffsets,
// after which the scatter kernel returns before touching the weights.
__global__ void k_tables32(const int64_t* __restrict__ hsc, const int64_t* __restrict__ wo, uint32_t T,
                           NoAllocScratch* s) {
  for (uint32_t t = threadIdx.x; t <= T; t += blockDim.x) {
    const int64_t v = hsc[t];
    bool bad = v < 0 || v > (int64_t)0xffffffffLL || (t == 0 && v != 0);
    if (t > 0) bad |= v <= hsc[t - 1];
    if (t < T) {
      const int64_t o = wo[t];
      bad |= o < 0 || (o & 3) != 0;
    }
    if (bad) {
      atomicOr(&s->ctl.err, kErrOffsets);
      atomicOr(&s->status, kErrOffsets);
    }
    s->hsc[t] = (uint32_t)v;
  }
}

}  // namespace
}  // namespace embbwd

using namespace embbwd;

extern "C" emb_status emb_nobag_bwd_sgd_atomic_noalloc(
    int device, int32_t T, const int64_t* hash_size_cumsum, const int64_t* weights_offsets,
    int32_t D, float* weights, const int64_t* indices, const int64_t* offsets, int64_t N,
    int32_t B, const void* grad_output, emb_dtype grad_dtype, float lr, uint32_t* device_status,
    void* stream) {
  if (device < 0 || device >= kNoAllocMaxDevices) return EMB_ERR_INVALID_ARG;
  if (T <= 0 || T > kMaxT || B <= 0 || (int64_t)B * T >= ((int64_t)1 << 31)) return EMB_ERR_INVALID_ARG;
  if (D <= 0 || D % 4 != 0 || D > 4096) return EMB_ERR_INVALID_ARG;
  if (N < 0 || N > kNoAllocMaxN) return EMB_ERR_INVALID_ARG;
  if (grad_dtype < EMB_F32 || grad_dtype > EMB_BF16) return EMB_ERR_INVALID_ARG;
  if (!hash_size_cumsum || !weights_offsets || !weights || !indices || !offsets || !grad_output)
    return EMB_ERR_INVALID_ARG;
  const size_t gvec = grad_dtype == EMB_F32 ? 16 : 8;
  if (reinterpret_cast<uintptr_t>(weights) % 16 || reinterpret_cast<uintptr_t>(grad_output) % gvec ||
      reinterpret_cast<uintptr_t>(indices) % 8 || reinterpret_cast<uintptr_t>(offsets) % 8 ||
      reinterpret_cast<uintptr_t>(device_status) % 4)
    return EMB_ERR_INVALID_ARG;

  int prev = -1;
  if (cudaGetDevice(&prev) != cudaSuccess) prev = -1;
  if (cudaSetDevice(device) != cudaSuccess) return EMB_ERR_INVALID_ARG;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  NoAllocScratch* sc = nullptr;
  cudaError_t e = scratch_address(device, &sc);
  if (e == cudaSuccess) e = cudaMemsetAsync(sc, 0, offsetof(NoAllocScratch, hsc), s);
  if (e == cudaSuccess && N > 0) {
    k_tables32<<<1, kThreads, 0, s>>>(hash_size_cumsum, weights_offsets, (uint32_t)T, sc);
    e = cudaGetLastError();
    DecodeArgs d;
    d.indices = indices;
    d.offsets = offsets;
    d.psw = nullptr;
    d.hsc = sc->hsc;
    d.N = N;
    d.B = (uint32_t)B;
    d.T = (uint32_t)T;
    d.BT = (uint32_t)B * (uint32_t)T;
    d.invB = 1.0f / (float)B;
    d.mean = 0;
    // index range and CSR checks (no radix histogram), then the atomic scatter,
    // which does nothing if a check failed
    HistArgs ha{d, &sc->ctl, &sc->status, 0, (int)sort_tile_for(N), nullptr, nullptr};
    if (e == cudaSuccess) e = launch_hist(ha, -1, T, s, false);
    AtomicArgs aa{d, &sc->ctl, &sc->status, grad_output, weights, weights_offsets, (uint32_t)D, lr};
    if (e == cudaSuccess) e = launch_nobag_atomic(aa, (int)grad_dtype, T, s, false);
  }
  if (e == cudaSuccess && device_status)
    e = cudaMemcpyAsync(device_status, &sc->status, sizeof(uint32_t), cudaMemcpyDeviceToDevice, s);
  if (prev >= 0) cudaSetDevice(prev);
  if (e != cudaSuccess) {
    cudaGetLastError();
    return EMB_ERR_CUDA;
  }
  return EMB_OK;
}
