// Range copies between page-locked host memory and HBM for the host-buffer
// exchange calls. The SMs move the data themselves (the host buffer is
// mapped into the device's address space), so one launch covers every
// domain's range, where the copy engines would need one call per range.
#include <cstdint>

#include "hx_host.h"

namespace hx {
namespace {

constexpr int kCopyThreads = 256;

// One block per chunk. When source and destination share their address
// mod 16, the chunk's aligned middle moves in 16-byte words, four per thread
// in flight; the few words around it, and every word otherwise, one by one.
__global__ void __launch_bounds__(kCopyThreads) k_copy_chunks(const float* __restrict__ src, float* __restrict__ dst,
                                                              const CopyChunk* __restrict__ chunks, int mode) {
  const CopyChunk c = chunks[blockIdx.x];
  const float* s = src + (mode == kCopyUnpack ? c.packed : c.word);
  float* d = dst + (mode == kCopyPack ? c.packed : c.word);
  const int n = c.n;
  const int t = static_cast<int>(threadIdx.x);
  const uintptr_t sa = reinterpret_cast<uintptr_t>(s), da = reinterpret_cast<uintptr_t>(d);
  if (((sa ^ da) & 15u) != 0) {
    for (int i = t; i < n; i += kCopyThreads) d[i] = s[i];
    return;
  }
  int head = static_cast<int>(((16u - (da & 15u)) & 15u) / 4u);
  if (head > n) head = n;
  const int nv = (n - head) / 4;   // 16-byte words in the middle
  const int4* sv = reinterpret_cast<const int4*>(s + head);
  int4* dv = reinterpret_cast<int4*>(d + head);
  int i = t;
  for (; i + 3 * kCopyThreads < nv; i += 4 * kCopyThreads) {
    const int4 a = sv[i], b = sv[i + kCopyThreads], e = sv[i + 2 * kCopyThreads], f = sv[i + 3 * kCopyThreads];
    dv[i] = a;
    dv[i + kCopyThreads] = b;
    dv[i + 2 * kCopyThreads] = e;
    dv[i + 3 * kCopyThreads] = f;
  }
  for (; i < nv; i += kCopyThreads) dv[i] = sv[i];
  if (t < head) d[t] = s[t];
  const int tail0 = head + 4 * nv;
  if (tail0 + t < n) d[tail0 + t] = s[tail0 + t];   // at most 3 words
}

}  // namespace

cudaError_t launch_copy_chunks(const float* src, float* dst, const CopyChunk* chunks, int n_chunks, int mode,
                               cudaStream_t s) {
  if (n_chunks <= 0) return cudaSuccess;
  k_copy_chunks<<<n_chunks, kCopyThreads, 0, s>>>(src, dst, chunks, mode);
  return cudaGetLastError();
}

}  // namespace hx
