// nm_layout.cuh -- operand images in the UMMA K-major swizzled layout.
//
// An "image" holds `rows` rows of a K-wide FP16 operand (a weight matrix
// W_l[N][K], or a 128-row activation tile [128][K]). K is cut from k = 0
// upward into segments of 64 columns (128-byte swizzle) while at least 64
// remain, then one of 32 (64-byte swizzle), then one of 16 (32-byte swizzle).
// Each segment starts 1024-byte aligned and stores row r at r * 2w bytes; the
// 16-byte chunk holding columns [8c, 8c+8) of a row is placed at the address
// XOR-swizzled by bits [7,10) of the plain offset, which is exactly the
// pattern a TMA copy with the matching CU_TENSOR_MAP_SWIZZLE_{128,64,32}B mode
// produces and that the tcgen05 shared-memory descriptor with swizzle mode
// {2, 4, 6} expects (8-row core-matrix groups 16w bytes apart).
//
// The packed weight blob is the sequence of per-layer weight images (each
// 1024-aligned) followed by the FP16 biases of all layers.
#pragma once

#include <cstdint>

namespace nm {

constexpr int kMaxLayers = 16;
constexpr int kMaxDim = 256;
constexpr int kTileM = 128;

__host__ __device__ __forceinline__ uint32_t align1024(uint32_t v) {
  return (v + 1023u) & ~1023u;
}

// Swizzle mode field of the tcgen05 smem descriptor for a segment width.
__host__ __device__ __forceinline__ uint32_t swizzle_code(int w) {
  return w == 64 ? 2u : (w == 32 ? 4u : 6u);
}

// Index of the tensor map (0: 128B, 1: 64B, 2: 32B swizzle) for a width.
__host__ __device__ __forceinline__ int swizzle_kind(int w) {
  return w == 64 ? 0 : (w == 32 ? 1 : 2);
}

// Plain byte offset p inside a segment of width w -> stored offset.
__host__ __device__ __forceinline__ uint32_t swz(uint32_t p, int w) {
  const uint32_t m = w == 64 ? 7u : (w == 32 ? 3u : 1u);
  return p ^ (((p >> 7) & m) << 4);
}

// Segment holding column k of a K-wide image with `rows` rows: its byte
// offset inside the image, its width and first column.
__host__ __device__ __forceinline__ void locate(uint32_t rows, int K, int k, uint32_t& seg_off,
                                                int& w, int& k0) {
  const int n64 = K >> 6;
  const int rem = K & 63;
  const uint32_t b64 = align1024(rows * 128u);
  if (k < (n64 << 6)) {
    w = 64;
    k0 = k & ~63;
    seg_off = static_cast<uint32_t>(k >> 6) * b64;
  } else if (rem >= 32 && k < (n64 << 6) + 32) {
    w = 32;
    k0 = n64 << 6;
    seg_off = static_cast<uint32_t>(n64) * b64;
  } else {
    w = 16;
    k0 = (n64 << 6) + (rem >= 32 ? 32 : 0);
    seg_off = static_cast<uint32_t>(n64) * b64 + (rem >= 32 ? align1024(rows * 64u) : 0u);
  }
}

// Number of segments of a K-wide image and their (width, first column).
__host__ __device__ __forceinline__ int segments(int K, int* w, int* k0) {
  int n = 0, k = 0;
  while (K - k >= 64) { w[n] = 64; k0[n++] = k; k += 64; }
  if (K - k >= 32) { w[n] = 32; k0[n++] = k; k += 32; }
  if (K - k >= 16) { w[n] = 16; k0[n++] = k; k += 16; }
  return n;
}

// Bytes spanned by an image (end of its last segment).
__host__ __device__ __forceinline__ uint32_t image_bytes(uint32_t rows, int K) {
  int w[16], k0[16];
  const int ns = segments(K, w, k0);
  uint32_t off = 0;
  for (int s = 0; s < ns; ++s) {
    off = align1024(off);
    off += rows * 2u * static_cast<uint32_t>(w[s]);
  }
  return off;
}

// Shared-memory matrix descriptor (tcgen05 format): start address >> 4 in bits
// [0,14), leading byte offset >> 4 in [16,30) (unused by the swizzled K-major
// layouts used here; set to 1), stride byte offset >> 4 in [32,46) (distance
// between consecutive 8-row core-matrix groups, 16w bytes for a w-wide
// segment), the fixed version field 1 at bit 46, base offset 0, and the
// swizzle mode in [61,64): 2 = 128-byte, 4 = 64-byte, 6 = 32-byte.
// A descriptor built from an offset relative to some 1024-aligned base becomes
// absolute by adding base >> 4 (the start field never carries past bit 13 for
// addresses inside the 228 KB shared window).
__host__ __device__ __forceinline__ uint64_t smem_desc(uint32_t saddr, uint32_t sbo_bytes,
                                                       uint32_t swizzle_code) {
  uint64_t d = 0;
  d |= static_cast<uint64_t>((saddr & 0x3FFFFu) >> 4);
  d |= static_cast<uint64_t>(1u) << 16;
  d |= static_cast<uint64_t>((sbo_bytes >> 4) & 0x3FFFu) << 32;
  d |= static_cast<uint64_t>(1u) << 46;
  d |= static_cast<uint64_t>(swizzle_code & 7u) << 61;
  return d;
}

// Instruction descriptor for kind::f16 with FP16 A and B, FP32 accumulator,
// both operands K-major, dense: D format in bits [4,6) = 1 (F32), A/B formats
// [7,10)/[10,13) = 0 (F16), N >> 3 in [17,23), M >> 4 in [24,29).
__host__ __device__ __forceinline__ uint32_t idesc_f16_f32(uint32_t M, uint32_t N) {
  return (1u << 4) | ((N >> 3) << 17) | ((M >> 4) << 24);
}

}  // namespace nm
