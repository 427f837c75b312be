// fa_common.cuh -- pieces shared by the forward (fa_fwd_sm103.cu) and backward
// (fa_bwd_sm103.cu) translation units: the device status word and the bounded
// mbarrier waits that set it, the TMA descriptor encoder, and host-side argument
// helpers.  Everything here sits in an unnamed namespace on purpose: each translation
// unit gets its own copy, in particular its own status word, and fa_status() reads
// and ORs the words of both.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>

#include <algorithm>
#include <cmath>
#include <cstdint>
#include <cstring>
#include <mutex>

#include "fa_gb300.h"
#include "sm103_ptx.cuh"

namespace fa {
namespace {

__device__ unsigned int g_status;

// Bounded mbarrier waits.  `wait` gives up when the CTA's abort flag is set or
// the deadline passes (then it sets the flag and the device status word);
// `drain` ignores the abort flag (used to wait for in-flight work on the way out).
struct Waiter {
  volatile uint32_t* abort_flag;
  unsigned long long timeout_ns;

  __device__ __forceinline__ bool wait(uint32_t bar, uint32_t parity) const {
    if (ptx::mbar_try_wait(bar, parity)) return true;
    return slow(bar, parity, true);
  }
  __device__ __forceinline__ bool drain(uint32_t bar, uint32_t parity) const {
    if (ptx::mbar_try_wait(bar, parity)) return true;
    return slow(bar, parity, false);
  }
  __device__ __forceinline__ bool slow(uint32_t bar, uint32_t parity, bool honour_abort) const {
    const uint64_t t0 = ptx::globaltimer_ns();
    while (true) {
#pragma unroll 1
      for (int i = 0; i < 16; ++i)
        if (ptx::mbar_try_wait(bar, parity)) return true;
      if (honour_abort && *abort_flag) return false;
      if (ptx::globaltimer_ns() - t0 > timeout_ns) {
        *abort_flag = 1u;
        atomicOr(&g_status, FA_STATUS_TIMEOUT);
        return false;
      }
    }
  }
};

// ---------------------------------------------------------------- host helpers
constexpr int kMaxDevices = 64;
constexpr unsigned long long kDefaultTimeoutNs = 2000000000ull;  // 2 s per wait

typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                  const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                  const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                  CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn() {
  static EncodeTiledFn fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* f = nullptr;
    cudaDriverEntryPointQueryResult q{};
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiledFn>(f);
  });
  return fn;
}

// [heads, rows, d] bf16 viewed as 3-D; box = 64 columns (128 bytes) x 128 rows x 1 head.
bool encode_map(CUtensorMap* m, const void* base, int heads, int rows, int d) {
  EncodeTiledFn fn = encode_fn();
  if (!fn) return false;
  const cuuint64_t dims[3] = {static_cast<cuuint64_t>(d), static_cast<cuuint64_t>(rows),
                              static_cast<cuuint64_t>(heads)};
  const cuuint64_t strides[2] = {static_cast<cuuint64_t>(d) * 2, static_cast<cuuint64_t>(rows) * d * 2};
  const cuuint32_t box[3] = {64, 128, 1};
  const cuuint32_t estr[3] = {1, 1, 1};
  return fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(base), dims, strides, box, estr,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// [heads, rows, row_bytes] bytes viewed as 3-D; box = 128 bytes x 128 rows x 1 head.
bool encode_map_u8(CUtensorMap* m, const void* base, int heads, int rows, int row_bytes) {
  EncodeTiledFn fn = encode_fn();
  if (!fn) return false;
  const cuuint64_t dims[3] = {static_cast<cuuint64_t>(row_bytes), static_cast<cuuint64_t>(rows),
                              static_cast<cuuint64_t>(heads)};
  const cuuint64_t strides[2] = {static_cast<cuuint64_t>(row_bytes),
                                 static_cast<cuuint64_t>(rows) * static_cast<cuuint64_t>(row_bytes)};
  const cuuint32_t box[3] = {128, 128, 1};
  const cuuint32_t estr[3] = {1, 1, 1};
  return fn(m, CU_TENSOR_MAP_DATA_TYPE_UINT8, 3, const_cast<void*>(base), dims, strides, box, estr,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// FA_OK when device `dev` is compute capability 10.3, FA_ERR_ARCH when it is not.
int check_arch(int dev) {
  int major = 0, minor = 0;
  if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess)
    return FA_ERR_CUDA;
  return (major == 10 && minor == 3) ? FA_OK : FA_ERR_ARCH;
}

bool is_device_pointer(const void* ptr) {
  cudaPointerAttributes a{};
  if (cudaPointerGetAttributes(&a, ptr) != cudaSuccess) {
    cudaGetLastError();
    return false;
  }
  return a.type == cudaMemoryTypeDevice || a.type == cudaMemoryTypeManaged;
}

bool overlaps(const void* a, size_t na, const void* b, size_t nb) {
  const uintptr_t x = reinterpret_cast<uintptr_t>(a), y = reinterpret_cast<uintptr_t>(b);
  return na > 0 && nb > 0 && x < y + nb && y < x + na;
}

size_t align256(size_t x) { return (x + 255) & ~static_cast<size_t>(255); }

// ---- host-to-host pipelines (fa_fwd_host, fa_bwd_host)
// Per device: one stream for host-to-device copies, one for device-to-host copies, two for
// the chunks' kernels (a causal chunk's longest CTA sets its kernel's duration however few
// heads it holds, so consecutive chunks run side by side on the SMs), and a pool of events;
// created on first use and kept until the process exits.  The mutex serialises the
// enqueueing of whole calls, so that two host threads never interleave their records of
// the shared events.
constexpr int kMaxChunks = 64;
// Default chunking.  When the host link binds (its copies take longer than the attention),
// at most seven chunks with the boundaries at 8, 14, 20, 25, 29, 31 and 32 thirty-seconds of
// the groups (rounded; empty chunks dropped): 32 groups give 8, 6, 6, 5, 4, 2, 1.  Large early
// chunks keep the link busy with few launches; small late ones shorten the tail (the last
// chunk's kernel and its copy back), which no later copy hides.  When the attention binds,
// eight equal chunks: a small last chunk would add the length of its longest causal CTA.
// The link time is estimated with the rate measured on GB300, about 200 GB/s per direction;
// the caller gives its kernels' time.  (Forward, causal N = 8192, d = 128, 32 groups: 1.22 ms
// against 1.27 ms with equal chunks; causal N = 32768: 6.6 against 7.1 ms the other way round.)
constexpr double kHostLinkBytesPerSec = 2.0e11;
constexpr double kForwardFlopsPerSec = 1.3e15;   // the forward kernel, measured
constexpr double kBackwardFlopsPerSec = 0.85e15;  // the backward's three kernels, measured
int default_chunks(int groups, double copy_bytes, double kernel_seconds, int (&sizes)[kMaxChunks]) {
  int n = 0;
  if (kernel_seconds >= 0.8 * copy_bytes / kHostLinkBytesPerSec) {
    const int per = (groups + 7) / 8;
    for (int g = 0; g < groups; g += per) sizes[n++] = std::min(per, groups - g);
    return n;
  }
  constexpr int kBounds[7] = {8, 14, 20, 25, 29, 31, 32};
  int prev = 0;
  for (int i = 0; i < 7; ++i) {
    const int b = static_cast<int>((static_cast<long long>(groups) * kBounds[i] + 16) / 32);
    if (b > prev) sizes[n++] = b - prev;
    prev = b;
  }
  return n;
}
// Chunk sizes: groups_per_chunk each (capped at kMaxChunks chunks), or the default above.
int chunk_sizes(int groups, int groups_per_chunk, double copy_bytes, double kernel_seconds,
                int (&sizes)[kMaxChunks]) {
  if (groups_per_chunk <= 0) return default_chunks(groups, copy_bytes, kernel_seconds, sizes);
  int per = groups_per_chunk, n = 0;
  if ((groups + per - 1) / per > kMaxChunks) per = (groups + kMaxChunks - 1) / kMaxChunks;
  for (int g = 0; g < groups; g += per) sizes[n++] = std::min(per, groups - g);
  return n;
}
constexpr int kComputeStreams = 2;
struct HostPipe {
  cudaStream_t in = nullptr, out = nullptr, comp[kComputeStreams] = {};
  cudaEvent_t start = nullptr, done = nullptr, loaded[kMaxChunks] = {}, computed[kMaxChunks] = {};
  std::mutex mu;
  bool ready = false;
};
HostPipe g_pipe[kMaxDevices];

int host_pipe(int dev, HostPipe** out) {
  HostPipe& hp = g_pipe[dev];
  if (!hp.ready) {
    const unsigned flags = cudaEventDisableTiming;
    for (int i = 0; i < kComputeStreams; ++i)
      if (cudaStreamCreateWithFlags(&hp.comp[i], cudaStreamNonBlocking) != cudaSuccess) return FA_ERR_CUDA;
    if (cudaStreamCreateWithFlags(&hp.in, cudaStreamNonBlocking) != cudaSuccess ||
        cudaStreamCreateWithFlags(&hp.out, cudaStreamNonBlocking) != cudaSuccess ||
        cudaEventCreateWithFlags(&hp.start, flags) != cudaSuccess ||
        cudaEventCreateWithFlags(&hp.done, flags) != cudaSuccess)
      return FA_ERR_CUDA;
    for (int c = 0; c < kMaxChunks; ++c)
      if (cudaEventCreateWithFlags(&hp.loaded[c], flags) != cudaSuccess ||
          cudaEventCreateWithFlags(&hp.computed[c], flags) != cudaSuccess)
        return FA_ERR_CUDA;
    hp.ready = true;
  }
  *out = &hp;
  return FA_OK;
}

bool is_pinned_host(const void* ptr) {
  cudaPointerAttributes attr{};
  if (cudaPointerGetAttributes(&attr, ptr) != cudaSuccess) {
    cudaGetLastError();
    return false;
  }
  return attr.type == cudaMemoryTypeHost;
}


}  // namespace
}  // namespace fa
