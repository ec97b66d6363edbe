// Copies between a caller's page-locked host buffer and a device buffer of
// the same slot layout, range by range (hx_host.cu). Used by the host-buffer
// exchange calls: home slots in, halo slots (coordinates) or home slots
// (forces) out.
#pragma once

#include <cstdint>

#include <cuda_runtime.h>

namespace hx {

// A piece of one range of 32-bit words, at most kCopyChunkWords long; one
// block copies one piece.
constexpr int kCopyChunkWords = 16384;   // 64 KB
struct CopyChunk {
  int64_t word;                           // first word (slot * 3 + component)
  int32_t n;                              // words, 1..kCopyChunkWords
  int32_t pad;
};
static_assert(sizeof(CopyChunk) == 16, "copy chunk must stay 16 bytes");

// dst[c.word + i] = src[c.word + i] for every chunk c and i < c.n. src and
// dst are device addresses (a mapped host buffer's device address included).
cudaError_t launch_copy_chunks(const float* src, float* dst, const CopyChunk* chunks, int n_chunks, cudaStream_t s);

}  // namespace hx
