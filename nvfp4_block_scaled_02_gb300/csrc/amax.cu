// amax.cu -- per-slice global amax of a bf16 tensor (the FP32 outer scale's
// input; End-to-End 4-Bit Training, "Low-precision formats on Blackwell";
// current vs periodic tensor scaling in the UE5M3 blog).
//
// Pure read stream: 128-bit loads, |x| as the integer bf16 pattern & 0x7FFF
// (the ordering of non-negative floats is the ordering of their bits), packed
// u16x2 max, a warp max (redux), a CTA max, and one atomicMax per CTA on the
// fp32 bit pattern of the result (after a zeroing kernel), or, with a
// caller's workspace, one launch whose last CTA per slice writes the result.
// MAX is exact and order-free, so the result does not depend on the schedule.
#include <atomic>

#include "device.cuh"
#include "launch.h"

namespace nvfp4 {

namespace {

constexpr int kThreads = 256;
constexpr int kUnroll = 4;

// The CTA's part of one slice's max |x| as a bf16 bit pattern (in thread 0;
// the other threads return garbage), from 128-bit streaming loads.
__device__ __forceinline__ uint32_t cta_absmax(const uint16_t* __restrict__ base, int64_t n) {
  const int64_t head0 = ((16 - ((uintptr_t)base & 15)) & 15) / 2;
  const int64_t head = head0 < n ? head0 : n;
  const uint4* v = reinterpret_cast<const uint4*>(base + head);
  const int64_t nvec = (n - head) / 8;
  const int64_t tail0 = head + nvec * 8;

  uint32_t m = 0;
  if (blockIdx.x == 0) {
    for (int64_t i = threadIdx.x; i < head; i += kThreads) m = max(m, (uint32_t)(base[i] & 0x7FFFu));
    for (int64_t i = tail0 + threadIdx.x; i < n; i += kThreads)
      m = max(m, (uint32_t)(base[i] & 0x7FFFu));
  }
  const int64_t stride = (int64_t)gridDim.x * kThreads;
  for (int64_t i = (int64_t)blockIdx.x * kThreads + threadIdx.x; i < nvec; i += stride * kUnroll) {
    uint4 r[kUnroll];
#pragma unroll
    for (int u = 0; u < kUnroll; ++u) {
      const int64_t j = i + u * stride;
      r[u] = j < nvec ? __ldcs(v + j) : make_uint4(0, 0, 0, 0);
    }
#pragma unroll
    for (int u = 0; u < kUnroll; ++u) m = max(m, absmax_bits4(r[u]));
  }
  m = __reduce_max_sync(0xFFFFFFFFu, m);
  __shared__ uint32_t wmax[kThreads / 32];
  if ((threadIdx.x & 31) == 0) wmax[threadIdx.x >> 5] = m;
  __syncthreads();
  if (threadIdx.x == 0)
    for (int w = 1; w < kThreads / 32; ++w) m = max(m, wmax[w]);
  return m;
}

__global__ void __launch_bounds__(kThreads) amax_kernel(const uint16_t* __restrict__ x, int64_t n,
                                                        uint32_t* amax_bits, int32_t* status) {
  pdl_begin();
  const uint32_t m = cta_absmax(x + blockIdx.y * n, n);
  if (threadIdx.x == 0) {
    if (m >= 0x7F80u) flag(status, NVFP4_DEV_NONFINITE_INPUT_BIT);
    if (m) atomicMax(amax_bits + blockIdx.y, m << 16);
  }
}

// The same in one launch, without a zeroed output: each CTA folds its maximum
// into workspace word 2s with an atomic max, makes that visible, and takes a
// ticket from word 2s + 1; the CTA holding the slice's last ticket reads the
// maximum back (an atomic exchange, so it sees every other CTA's), writes
// amax[s] and returns both words to zero for the next call. No CTA waits.
__global__ void __launch_bounds__(kThreads) amax_ticket_kernel(const uint16_t* __restrict__ x,
                                                               int64_t n, float* amax,
                                                               uint32_t* ws, int32_t* status) {
  pdl_begin();
  const uint32_t m = cta_absmax(x + blockIdx.y * n, n);
  if (threadIdx.x == 0) {
    uint32_t* w = ws + 2 * blockIdx.y;
    if (m >= 0x7F80u) flag(status, NVFP4_DEV_NONFINITE_INPUT_BIT);
    if (m) atomicMax(w, m);
    __threadfence();
    if (atomicAdd(w + 1, 1u) == gridDim.x - 1) {
      const uint32_t v = atomicExch(w, 0u);
      atomicExch(w + 1, 0u);
      amax[blockIdx.y] = __uint_as_float(v << 16);
    }
  }
}

// Zeroes n 32-bit words (the amax output before its atomic max, 4/6 bitmaps
// before their atomic ORs): a kernel of our own, launched like every other so
// that it overlaps the previous kernel's tail, where a memset would not.
__global__ void zero_words_kernel(uint32_t* p, int64_t n) {
  pdl_begin();
  const int64_t stride = (int64_t)gridDim.x * blockDim.x;
  for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < n; i += stride) p[i] = 0u;
}

}  // namespace

cudaError_t launch_zero_words(uint32_t* p, int64_t n, cudaStream_t st) {
  if (n <= 0) return cudaSuccess;
  const int64_t want = (n + 255) / 256, cap = (int64_t)sm_count() * 4;
  return launch_pdl(zero_words_kernel, dim3((unsigned)(want < cap ? want : cap)), dim3(256), st, p,
                    n);
}

// Grid of the amax kernels: CTAs per slice, enough to fill the GPU.
static int64_t amax_ctas(int64_t S, int64_t n) {
  const int64_t nvec = n / 8 + 1;
  const int64_t want = (nvec + kThreads * kUnroll - 1) / (kThreads * kUnroll);
  const int64_t cap = std::max<int64_t>(1, (int64_t)sm_count() * 8 / std::max<int64_t>(1, S));
  return std::min(want, cap);
}

cudaError_t launch_amax_ticket(const uint16_t* x, int64_t S, int64_t n, float* amax,
                               uint32_t* ws, int32_t* status, cudaStream_t st) {
  const int64_t ctas = amax_ctas(S, n);
  for (int64_t s0 = 0; s0 < S; s0 += 65535) {
    dim3 grid((unsigned)ctas, (unsigned)std::min<int64_t>(S - s0, 65535));
    const cudaError_t e = launch_pdl(amax_ticket_kernel, grid, dim3(kThreads), st, x + s0 * n, n,
                                     amax + s0, ws + 2 * s0, status);
    if (e != cudaSuccess) return e;
  }
  return cudaSuccess;
}

cudaError_t launch_amax(const uint16_t* x, int64_t S, int64_t n, float* amax, int32_t* status,
                        cudaStream_t st) {
  cudaError_t e = launch_zero_words(reinterpret_cast<uint32_t*>(amax), S, st);  // for the atomic max
  if (e != cudaSuccess) return e;
  if (n == 0) return cudaSuccess;
  const int64_t ctas = amax_ctas(S, n);
  for (int64_t s0 = 0; s0 < S; s0 += 65535) {
    dim3 grid((unsigned)ctas, (unsigned)std::min<int64_t>(S - s0, 65535));
    e = launch_pdl(amax_kernel, grid, dim3(kThreads), st, x + s0 * n, n,
                   reinterpret_cast<uint32_t*>(amax + s0), status);
    if (e != cudaSuccess) return e;
  }
  return cudaSuccess;
}

// ---- the amax without any caller memory but its input and output ---------
// Some callers cannot allocate device memory: an operator hook inside another
// framework that hands out no workspace, a serving or real-time loop that
// fixes all its memory at start-up, code that must not call cudaMalloc or
// cudaFree because those can synchronise the device. For them the one-launch
// amax takes its two scratch words per slice from a fixed array in this
// library's own device image (every GPU that loads the library holds it until
// the process exits). In host code the array's name is only a stand-in, not
// a device address: its address is looked up once per device.
static __device__ __align__(256) uint32_t g_amax_scratch[2 * kAmaxNoAllocMaxSlices];
static std::atomic<uint32_t*> g_amax_scratch_at[64];  // its device address, per device

cudaError_t launch_amax_noalloc(const uint16_t* x, int64_t S, int64_t n, float* amax,
                                int32_t* status, cudaStream_t st) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
  uint32_t* ws = g_amax_scratch_at[dev].load(std::memory_order_acquire);
  if (ws == nullptr) {  // first call on this device (that device is current)
    void* p = nullptr;
    e = cudaGetSymbolAddress(&p, g_amax_scratch);
    if (e != cudaSuccess) return e;
    ws = static_cast<uint32_t*>(p);
    g_amax_scratch_at[dev].store(ws, std::memory_order_release);
  }
  // the words of this call's slices start at zero whatever an earlier call
  // (one that overlapped another on the GPU, say) left in them
  e = launch_zero_words(ws, 2 * S, st);
  if (e != cudaSuccess) return e;
  return launch_amax_ticket(x, S, n, amax, ws, status, st);
}

}  // namespace nvfp4
