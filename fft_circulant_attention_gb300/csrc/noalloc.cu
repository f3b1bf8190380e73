// cat_forward_noalloc: the short-sequence forward with its workspace in a
// fixed array of the library's device image instead of plan-owned
// cudaMalloc memory, for callers that cannot allocate device memory (their
// memory is owned by a caching or pooled allocator, or they cannot afford
// the device-wide synchronisation cudaMalloc/cudaFree imply).
//
// The kernels are the plan path's own (score, softmax + spectrum, circulant
// product); only the workspace pointers differ.  The array lives as long as
// the process, on every device that loads the library; every call shares it.
#include <cuda_runtime.h>

#include <cmath>
#include <cstdint>
#include <mutex>

#include "../../include/cat.h"
#include "cat_internal.h"

namespace {

constexpr size_t kAlign = 256;
constexpr size_t align_up(size_t x) { return (x + kAlign - 1) / kAlign * kAlign; }

// Regions of the workspace, in bytes from its start.
constexpr size_t kRows = (size_t)CAT_NOALLOC_MAX_ROWS;
constexpr size_t kOffZ2 = 0;                                             // float2 [B·H·N]
constexpr size_t kOffZs = align_up(kOffZ2 + kRows * sizeof(float2));     // float  [B·H·N]
constexpr size_t kOffZf = align_up(kOffZs + kRows * sizeof(float));      // float2 [B·H·N]
constexpr size_t kOffTw = align_up(kOffZf + kRows * sizeof(float2));     // float2 [N]
constexpr size_t kOffSt = align_up(kOffTw + CAT_NOALLOC_MAX_N * sizeof(float2));  // status
constexpr size_t kBytes = align_up(kOffSt + sizeof(unsigned int));

// The workspace.  In host code this name is only a handle for the runtime:
// its device address comes from cudaGetSymbolAddress, per device.
static __device__ __align__(256) unsigned char g_noalloc_ws[kBytes];

constexpr int kMaxDevices = 64;
struct DeviceState {
  unsigned char* base = nullptr;  // device address of g_noalloc_ws
  int sms = 0;                    // multiprocessors (launch shapes of the score kernels)
  int tw_n = 0;                   // length the twiddle region holds; 0 = none or refilling
};
DeviceState g_state[kMaxDevices];
std::mutex g_mutex;

// W[j] = exp(-2πi j/N) for j < N, evaluated in fp64 and rounded to fp32.
__global__ void fill_twiddles(float2* __restrict__ tw, int N) {
  for (int j = blockIdx.x * blockDim.x + threadIdx.x; j < N; j += gridDim.x * blockDim.x) {
    double s, c;
    sincospi(-2.0 * (double)j / (double)N, &s, &c);
    tw[j] = make_float2((float)c, (float)s);
  }
}

bool overlaps(const void* a, size_t na, const void* b, size_t nb) {
  uintptr_t x = (uintptr_t)a, y = (uintptr_t)b;
  return x < y + nb && y < x + na;
}

}  // namespace

extern "C" int cat_forward_noalloc(const void* X, const void* WA, const void* V, void* O, int B,
                                   int N, int D, int H, int dtype, void* stream) {
  int st = cat::validate(B, N, D, H, dtype);
  if (st != CAT_OK) return st;
  if (N > CAT_NOALLOC_MAX_N || (long long)B * H * N > (long long)CAT_NOALLOC_MAX_ROWS)
    return CAT_ERR_TOO_LARGE;
  if (B == 0) return CAT_OK;
  if (!X || !WA || !V || !O) return CAT_ERR_INVALID_ARG;
  if (((uintptr_t)X | (uintptr_t)WA | (uintptr_t)V | (uintptr_t)O) & 15) return CAT_ERR_MISALIGNED;
  const size_t es = dtype == CAT_BF16 ? 2 : 4;
  const size_t nx = (size_t)B * N * D * es, nw = (size_t)D * H * es;
  if (overlaps(O, nx, X, nx) || overlaps(O, nx, WA, nw) || overlaps(O, nx, V, nx))
    return CAT_ERR_ALIAS;

  // A plan on the stack: shape, launch configuration and workspace pointers,
  // no allocation.
  cat_plan_s p{};
  p.B = B; p.N = N; p.D = D; p.H = H; p.dtype = dtype;
  p.dh = D / H;
  p.npair = (p.dh + 1) / 2;
  p.stream = (cudaStream_t)stream;
  st = cat::configure_smem_path(&p);
  if (st != CAT_OK) return st;

  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return CAT_ERR_CUDA;
  p.device = dev;
  bool refill;
  unsigned char* base;
  {
    std::lock_guard<std::mutex> lock(g_mutex);
    DeviceState& ds = g_state[dev];
    if (!ds.base) {
      // One-time set-up on this device (it is current): the array's device
      // address and the multiprocessor count the score kernels size their
      // grids by.
      void* ptr = nullptr;
      int sms = 0;
      if (cudaGetSymbolAddress(&ptr, g_noalloc_ws) != cudaSuccess || !ptr ||
          cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess ||
          sms <= 0) {
        cudaGetLastError();
        return CAT_ERR_CUDA;
      }
      ds.base = (unsigned char*)ptr;
      ds.sms = sms;
    }
    base = ds.base;
    p.sms = ds.sms;
    refill = ds.tw_n != N;
    // While the region is being refilled it holds no valid length: a call
    // that fails before the fill is enqueued leaves it marked empty, so the
    // next call refills it.
    if (refill) ds.tw_n = 0;
  }
  p.z2 = (float2*)(base + kOffZ2);
  p.zs = (float*)(base + kOffZs);
  p.zf = (float2*)(base + kOffZf);
  p.tw = (float2*)(base + kOffTw);
  p.status = (unsigned int*)(base + kOffSt);

  cudaError_t e = cat::setup_score_kernels(&p);
  if (e == cudaSuccess) e = cat::setup_smem_kernels(&p);
  if (e != cudaSuccess) return CAT_ERR_CUDA;
  if (refill) {
    fill_twiddles<<<(N + 255) / 256, 256, 0, p.stream>>>(p.tw, N);
    if (cudaGetLastError() != cudaSuccess) return CAT_ERR_CUDA;
    std::lock_guard<std::mutex> lock(g_mutex);
    g_state[dev].tw_n = N;
  }
  // The status word keeps the previous call's value: clear it.
  if (cudaMemsetAsync(p.status, 0, sizeof(unsigned int), p.stream) != cudaSuccess)
    return CAT_ERR_CUDA;
  e = cat::launch_score(&p, X, WA);
  if (e == cudaSuccess) e = cat::launch_softmax_spectrum(&p);
  if (e == cudaSuccess) e = cat::launch_conv_smem(&p, V, O);
  return e == cudaSuccess ? CAT_OK : CAT_ERR_CUDA;
}
