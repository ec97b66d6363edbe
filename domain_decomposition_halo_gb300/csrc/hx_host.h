// Range copies of the host-buffer exchange calls (hx_host.cu): between a
// caller's page-locked host buffer and a device buffer of the same slot
// layout, range by range; and, for the packed calls, between the slot layout
// and the home or halo ranges laid end to end in one device buffer.
#pragma once

#include <cstdint>

#include <cuda_runtime.h>

namespace hx {

// A piece of one range of 32-bit words, at most kCopyChunkWords long; one
// block copies one piece. `word` is its place in the slot layout, `packed`
// its place in the ranges laid end to end (every domain's home range, or
// every domain's halo range, domain after domain).
constexpr int kCopyChunkWords = 16384;   // 64 KB
struct CopyChunk {
  int64_t word;                           // first word in the layout (slot * 3 + component)
  int64_t packed;                         // first word in the packed ranges
  int32_t n;                              // words, 1..kCopyChunkWords
  int32_t pad;
};
static_assert(sizeof(CopyChunk) == 24, "copy chunk must stay 24 bytes");

// How a launch of the range copies reads and writes.
enum CopyMode : int {
  kCopySame = 0,     // dst[word + i] = src[word + i]   (two buffers of the slot layout)
  kCopyPack = 1,     // dst[packed + i] = src[word + i] (layout -> packed ranges)
  kCopyUnpack = 2,   // dst[word + i] = src[packed + i] (packed ranges -> layout)
};

// One block per chunk, for every chunk c and i < c.n, as `mode` says. src and
// dst are device addresses (a mapped host buffer's device address included).
cudaError_t launch_copy_chunks(const float* src, float* dst, const CopyChunk* chunks, int n_chunks, int mode,
                               cudaStream_t s);

}  // namespace hx
