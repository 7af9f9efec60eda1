// nm_api.cu -- the C ABI of libnmmlp (declared in include/nm_mlp.h) and the
// weight pack/unpack kernels.
//
// Pack ("Profiling neural material inference", "Row-major versus
// InferencingOptimal weights": a one-time conversion of the canonical FP16
// row-major matrices into an opaque device layout) is a pure permutation:
// each thread moves one 16-byte chunk (8 weights of one row) from the
// row-major matrix to its swizzled place in the packed blob, and biases are
// copied unchanged behind the weight images. Unpack is the same map run
// backwards.
#include <cuda.h>
#include <cuda_fp8.h>
#include <cuda_runtime.h>
#include <cudaTypedefs.h>

#include <cstdint>
#include <cstring>
#include <mutex>
#include <new>

#include "nm_internal.h"
#include "nm_mlp.h"

namespace nm {

__global__ void __launch_bounds__(256) pack_kernel(const __grid_constant__ PackParams p, int unpack) {
  const uint32_t total_w = p.chunk_start[p.L];
  const uint32_t total = total_w + p.bias_chunk_start[p.L];
  for (uint32_t g = blockIdx.x * blockDim.x + threadIdx.x; g < total; g += gridDim.x * blockDim.x) {
    if (g < total_w) {
      int l = 0;
      while (g >= p.chunk_start[l + 1]) ++l;
      const uint32_t idx = g - p.chunk_start[l];
      const int K = p.dims[l], N = p.dims[l + 1], kc = K >> 3;
      const int n = static_cast<int>(idx / static_cast<uint32_t>(kc));
      const int col = static_cast<int>(idx - static_cast<uint32_t>(n * kc)) << 3;
      uint32_t off;
      int w, k0;
      locate(static_cast<uint32_t>(N), K, col, off, w, k0);
      const uint32_t dst =
          p.w_off[l] + off + swz(static_cast<uint32_t>(n * 2 * w + (col - k0) * 2), w);
      uint4* packed = reinterpret_cast<uint4*>(p.blob + dst);
      uint4* rowmajor = reinterpret_cast<uint4*>(p.rm_w[l] + static_cast<size_t>(n) * K + col);
      if (!unpack)
        *packed = __ldg(rowmajor);
      else
        *rowmajor = *packed;
    } else {
      const uint32_t gb = g - total_w;
      int l = 0;
      while (gb >= p.bias_chunk_start[l + 1]) ++l;
      uint4* packed = reinterpret_cast<uint4*>(p.blob + p.bias_off) + gb;
      uint4* rowmajor = reinterpret_cast<uint4*>(p.rm_b[l]) + (gb - p.bias_chunk_start[l]);
      if (!unpack)
        *packed = __ldg(rowmajor);
      else
        *rowmajor = *packed;
    }
  }
}

cudaError_t launch_pack(const PackParams& p, bool unpack, int num_sms, cudaStream_t stream) {
  const uint32_t total = p.chunk_start[p.L] + p.bias_chunk_start[p.L];
  int grid = static_cast<int>((total + 255u) / 256u);
  if (grid > 4 * num_sms) grid = 4 * num_sms;
  if (grid < 1) grid = 1;
  pack_kernel<<<grid, 256, 0, stream>>>(p, unpack ? 1 : 0);
  return cudaGetLastError();
}

// E4M3 images: thread g rounds the 16 FP16 weights W_l[n][col .. col + 15]
// -- two 16-byte chunks of the packed FP16 image -- to E4M3 and stores them
// as one 16-byte chunk. In the FP16-unit view of the E4M3 image (K/2 columns
// of 2 bytes), that chunk is the 8-column chunk at column col / 2.
__global__ void __launch_bounds__(256) pack_fp8_kernel(const __grid_constant__ PackParams p,
                                                       const __grid_constant__ Fp8Offsets o,
                                                       uint8_t* region) {
  const uint32_t total = o.chunk_start[p.L];
  for (uint32_t g = blockIdx.x * blockDim.x + threadIdx.x; g < total; g += gridDim.x * blockDim.x) {
    int l = 1;
    while (g >= o.chunk_start[l + 1]) ++l;
    const uint32_t idx = g - o.chunk_start[l];
    const int K = p.dims[l], N = p.dims[l + 1], kc = K >> 4;
    const int n = static_cast<int>(idx / static_cast<uint32_t>(kc));
    const int col = static_cast<int>(idx - static_cast<uint32_t>(n * kc)) << 4;
    uint32_t off;
    int w, k0;
    locate(static_cast<uint32_t>(N), K >> 1, col >> 1, off, w, k0);
    const uint32_t dst = o.off[l] + off + swz(static_cast<uint32_t>(n * 2 * w + (col - 2 * k0)), w);
    // the two source chunks (columns col and col + 8 lie in one FP16 segment)
    locate(static_cast<uint32_t>(N), K, col, off, w, k0);
    const uint32_t src = p.w_off[l] + off + swz(static_cast<uint32_t>(n * 2 * w + (col - k0) * 2), w);
    const uint32_t src2 =
        p.w_off[l] + off + swz(static_cast<uint32_t>(n * 2 * w + (col + 8 - k0) * 2), w);
    const uint4 a = *reinterpret_cast<const uint4*>(p.blob + src);
    const uint4 b = *reinterpret_cast<const uint4*>(p.blob + src2);
    const uint32_t hw[8] = {a.x, a.y, a.z, a.w, b.x, b.y, b.z, b.w};
    uint32_t q[4];
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      __half2_raw h0, h1;
      h0.x = static_cast<unsigned short>(hw[2 * j] & 0xFFFFu);
      h0.y = static_cast<unsigned short>(hw[2 * j] >> 16);
      h1.x = static_cast<unsigned short>(hw[2 * j + 1] & 0xFFFFu);
      h1.y = static_cast<unsigned short>(hw[2 * j + 1] >> 16);
      const uint32_t lo = __nv_cvt_halfraw2_to_fp8x2(h0, __NV_SATFINITE, __NV_E4M3);
      const uint32_t hi = __nv_cvt_halfraw2_to_fp8x2(h1, __NV_SATFINITE, __NV_E4M3);
      q[j] = lo | (hi << 16);
    }
    *reinterpret_cast<uint4*>(region + dst) = make_uint4(q[0], q[1], q[2], q[3]);
  }
}

uint32_t fp8_layout(const int32_t* dims, int L, uint32_t* off) {
  if (L < 2) return 0;
  for (int l = 1; l < L; ++l)
    if (dims[l] % 32 != 0) return 0;
  uint32_t o = 0;
  off[0] = 0;
  for (int l = 1; l < L; ++l) {
    o = align1024(o);
    off[l] = o;
    o += image_bytes(static_cast<uint32_t>(dims[l + 1]), dims[l] >> 1);
  }
  return o;
}

cudaError_t launch_pack_fp8(const PackParams& p, const uint32_t* fp8_off, uint8_t* region,
                            int num_sms, cudaStream_t stream) {
  Fp8Offsets o;
  std::memset(&o, 0, sizeof(o));
  uint32_t c = 0;
  for (int l = 1; l < p.L; ++l) {
    o.off[l] = fp8_off[l];
    o.chunk_start[l] = c;
    c += static_cast<uint32_t>(p.dims[l] * p.dims[l + 1] / 16);
  }
  o.chunk_start[p.L] = c;
  int grid = static_cast<int>((c + 255u) / 256u);
  if (grid > 4 * num_sms) grid = 4 * num_sms;
  if (grid < 1) grid = 1;
  pack_fp8_kernel<<<grid, 256, 0, stream>>>(p, o, region);
  return cudaGetLastError();
}

// ---------------------------------------------------------------- host helpers
namespace {

PFN_cuTensorMapEncodeTiled_v12000 g_encode = nullptr;
std::once_flag g_encode_once;

nm_status get_encoder() {
  std::call_once(g_encode_once, [] {
    void* fn = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      g_encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
  });
  return g_encode ? NM_OK : NM_ERR_CUDA;
}

// 2-D map over a row-major FP16 [rows][width] matrix; box = [box_rows][box_w]
// with the swizzle that matches a box_w-wide segment.
nm_status encode_map(CUtensorMap* m, const void* ptr, int width, int64_t rows, int box_w,
                     int box_rows) {
  cuuint64_t gdim[2] = {static_cast<cuuint64_t>(width), static_cast<cuuint64_t>(rows)};
  cuuint64_t gstride[1] = {static_cast<cuuint64_t>(width) * 2u};
  cuuint32_t box[2] = {static_cast<cuuint32_t>(box_w), static_cast<cuuint32_t>(box_rows)};
  cuuint32_t estride[2] = {1, 1};
  const CUtensorMapSwizzle sw = box_w == 64 ? CU_TENSOR_MAP_SWIZZLE_128B
                                : box_w == 32 ? CU_TENSOR_MAP_SWIZZLE_64B
                                              : CU_TENSOR_MAP_SWIZZLE_32B;
  const CUresult r = g_encode(m, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 2, const_cast<void*>(ptr), gdim,
                              gstride, box, estride, CU_TENSOR_MAP_INTERLEAVE_NONE, sw,
                              CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? NM_OK : NM_ERR_CUDA;
}

}  // namespace

nm_status check_dims(const int32_t* dims, int32_t n_dims) {
  if (!dims || n_dims < 2) return NM_ERR_INVALID_ARG;
  const int L = n_dims - 1;
  if (L > kMaxLayers) return NM_ERR_UNSUPPORTED;
  for (int l = 0; l <= L; ++l)
    if (dims[l] < 16 || dims[l] > kMaxDim || dims[l] % 16 != 0) return NM_ERR_UNSUPPORTED;
  return NM_OK;
}

size_t net_layout(const int32_t* dims, int L, FusedParams& p, uint32_t* w_off, uint32_t* rm_off,
                  uint32_t* rm_b_off, size_t* mirror_elems) {
  p.L = L;
  uint32_t off = 0;
  size_t rm = 0;
  for (int l = 0; l < L; ++l) {
    off = align1024(off);
    w_off[l] = off;
    off += image_bytes(static_cast<uint32_t>(dims[l + 1]), dims[l]);
    if (rm_off) rm_off[l] = static_cast<uint32_t>(rm);
    rm += static_cast<size_t>(dims[l]) * dims[l + 1];
  }
  for (int l = 0; l < L; ++l) {
    if (rm_b_off) rm_b_off[l] = static_cast<uint32_t>(rm);
    rm += static_cast<size_t>(dims[l + 1]);
  }
  if (mirror_elems) *mirror_elems = rm;
  p.bias_off = align1024(off);
  uint32_t nb = 0;
  for (int l = 0; l < L; ++l) nb += static_cast<uint32_t>(dims[l + 1]);
  return p.bias_off + 2u * nb;
}

void set_bias_params(const Schedule& sc, const int32_t* dims, int L, FusedParams& p) {
  uint32_t row0 = 0;
  for (int l = 0; l < L; ++l) {
    p.bias_row0[l] = row0;
    p.bslab_off[l] = sc.layer[l].bslab_off;
    row0 += static_cast<uint32_t>(dims[l + 1]);
  }
  p.n_bias = row0;
}

nm_status encode_io_maps(FusedParams& p, const int32_t* dims, int L, const void* in, void* out,
                         int64_t n) {
  nm_status st = get_encoder();
  if (st != NM_OK) return st;
  std::memset(p.tm_in, 0, sizeof(p.tm_in));
  std::memset(p.tm_out, 0, sizeof(p.tm_out));
  int w[16], k0[16];
  const int ns = segments(dims[0], w, k0);
  for (int s = 0; s < ns; ++s) {
    st = encode_map(&p.tm_in[swizzle_kind(w[s])], in, dims[0], n, w[s], kTileM);
    if (st != NM_OK) return st;
  }
  // Output: 32-row boxes of 32 columns (64-byte swizzle), plus 16 columns
  // (32-byte swizzle) for a trailing 16-column chunk.
  const int dl = dims[L];
  if (dl >= 32) {
    st = encode_map(&p.tm_out[swizzle_kind(32)], out, dl, n, 32, 32);
    if (st != NM_OK) return st;
  }
  if (dl & 31) {
    st = encode_map(&p.tm_out[swizzle_kind(16)], out, dl, n, 16, 32);
    if (st != NM_OK) return st;
  }
  return NM_OK;
}

PackParams make_pack_params(const int32_t* dims, int L, const uint32_t* w_off, uint32_t bias_off,
                            uint8_t* blob) {
  PackParams pp;
  std::memset(&pp, 0, sizeof(pp));
  pp.L = L;
  uint32_t cw = 0, cb = 0;
  for (int l = 0; l <= L; ++l) pp.dims[l] = dims[l];
  for (int l = 0; l < L; ++l) {
    pp.w_off[l] = w_off[l];
    pp.chunk_start[l] = cw;
    pp.bias_chunk_start[l] = cb;
    cw += static_cast<uint32_t>(dims[l] * dims[l + 1] / 8);
    cb += static_cast<uint32_t>(dims[l + 1] / 8);
  }
  pp.chunk_start[L] = cw;
  pp.bias_chunk_start[L] = cb;
  pp.bias_off = bias_off;
  pp.blob = blob;
  return pp;
}

}  // namespace nm

using nm::FusedParams;
using nm::PackParams;

struct nm_mlp {
  FusedParams params;  // kernel parameter block (offsets, tensor maps, plan)
  int L = 0;
  int32_t dims[nm::kMaxLayers + 1] = {};
  uint32_t w_off[nm::kMaxLayers] = {};   // byte offset of each layer's image in the blob
  uint32_t rm_off[nm::kMaxLayers] = {};  // element offset of each W_l in the mirror
  size_t blob_size = 0;
  uint8_t* blob = nullptr;       // packed weight images + FP16 biases (device)
  uint8_t* sched = nullptr;      // nm::Schedule (device)
  uint32_t* status = nullptr;    // device status word
  uint16_t* mirror = nullptr;    // row-major weights + biases for the row-major ablation
  uint32_t rm_b_off[nm::kMaxLayers] = {};
  size_t mirror_elems = 0;
  // E4M3 images of the narrow-precision variant: in the blob's allocation
  // from byte fp8_base on (fp8_size = 0: the network has none), with their
  // own schedule (the FP16-unit view: K/2 columns, the images' offsets).
  size_t fp8_base = 0;
  size_t fp8_size = 0;
  uint32_t fp8_off[nm::kMaxLayers] = {};
  uint8_t* sched8 = nullptr;
  bool fp8_valid = false;  // the images match the packed FP16 blob
  bool packed = false;
  bool mirror_valid = false;
  // A packing kernel (weights or the row-major mirror) was the last of this
  // handle's launches on `pack_stream`: the next dispatch there must not
  // overlap it, since the kernel reads the weights before its grid
  // dependency wait.
  bool pack_pending = false;
  cudaStream_t pack_stream = nullptr;
  int variant = nm::kVarFused;
  uint64_t wait_ns = 2000000000ull;
  uint32_t test_stall = 0;
  uint32_t test_check_cols = 0;  // checking build: lowered TMEM limit (0: none)
  int device = 0;
  int num_sms = 0;
  uint32_t smem_optin = 0;
  // I/O tensor maps of recent (in, out, n) triples, so that callers rotating
  // among a few buffer sets do not re-encode them on every dispatch.
  struct MapEntry {
    CUtensorMap tm_in[3];
    CUtensorMap tm_out[3];
    const void* in = nullptr;
    const void* out = nullptr;
    int64_t n = -1;
  };
  static constexpr int kMapCache = 16;
  MapEntry maps[kMapCache];
  int map_next = 0;
  // host-buffer pipeline (nm_mlp_infer_host)
  int64_t host_chunk = 0;              // rows per chunk requested (0: default)
  int64_t hs_rows = 0;                 // rows per chunk the staging buffers hold
  size_t hs_in_bytes = 0;              // input part of one staging buffer (256-aligned)
  size_t hs_each = 0;                  // bytes of one staging buffer
  uint8_t* hs_stage = nullptr;         // kHostStreams staging buffers (device)
  cudaStream_t hs[3] = {};
  cudaEvent_t hs_start = nullptr;
  cudaEvent_t hs_done[3] = {};
};

namespace {

using nm::aligned16;
using nm::kMaxRows;

constexpr int kHostStreams = 3;

// I/O tensor maps for (in, out, n), from the handle's cache of recent
// triples when possible.
nm_status cached_io_maps(nm_mlp* h, const void* in, void* out, int64_t n) {
  FusedParams& p = h->params;
  for (int i = 0; i < nm_mlp::kMapCache; ++i) {
    const nm_mlp::MapEntry& e = h->maps[i];
    if (e.in == in && e.out == out && e.n == n) {
      std::memcpy(p.tm_in, e.tm_in, sizeof(p.tm_in));
      std::memcpy(p.tm_out, e.tm_out, sizeof(p.tm_out));
      return NM_OK;
    }
  }
  const nm_status st = nm::encode_io_maps(p, h->dims, h->L, in, out, n);
  if (st != NM_OK) return st;
  nm_mlp::MapEntry& e = h->maps[h->map_next];
  h->map_next = (h->map_next + 1) % nm_mlp::kMapCache;
  std::memcpy(e.tm_in, p.tm_in, sizeof(p.tm_in));
  std::memcpy(e.tm_out, p.tm_out, sizeof(p.tm_out));
  e.in = in;
  e.out = out;
  e.n = n;
  return NM_OK;
}

PackParams make_pack_params(const nm_mlp* h) {
  return nm::make_pack_params(h->dims, h->L, h->w_off, h->params.bias_off, h->blob);
}

// The E4M3 images, converted from the packed FP16 blob on `stream` the first
// time the narrow-precision variant needs them after a pack.
// A one-time conversion the caller did not ask for must not end up only in a
// graph being captured (the handle would count it as done before any replay):
// such a dispatch is refused while `stream` captures.
bool capturing(cudaStream_t stream) {
  cudaStreamCaptureStatus cs = cudaStreamCaptureStatusNone;
  return cudaStreamIsCapturing(stream, &cs) != cudaSuccess || cs != cudaStreamCaptureStatusNone;
}

nm_status ensure_fp8(nm_mlp* h, cudaStream_t stream, bool in_pack = false) {
  if (h->fp8_valid) return NM_OK;
  if (!in_pack && capturing(stream)) return NM_ERR_UNSUPPORTED;
  if (nm::launch_pack_fp8(make_pack_params(h), h->fp8_off, h->blob + h->fp8_base, h->num_sms,
                          stream) != cudaSuccess)
    return NM_ERR_CUDA;
  h->pack_pending = true;
  h->pack_stream = stream;
  h->fp8_valid = true;
  return NM_OK;
}

nm_status ensure_mirror(nm_mlp* h, cudaStream_t stream) {
  if (h->mirror_valid) return NM_OK;
  if (capturing(stream)) return NM_ERR_UNSUPPORTED;
  if (!h->mirror) {
    if (cudaMalloc(&h->mirror, h->mirror_elems * sizeof(uint16_t)) != cudaSuccess) {
      h->mirror = nullptr;
      return NM_ERR_OOM;
    }
  }
  PackParams pp = make_pack_params(h);
  for (int l = 0; l < h->L; ++l) {
    pp.rm_w[l] = h->mirror + h->rm_off[l];
    pp.rm_b[l] = h->mirror + h->rm_b_off[l];
  }
  if (nm::launch_pack(pp, true, h->num_sms, stream) != cudaSuccess) return NM_ERR_CUDA;
  h->pack_pending = true;
  h->pack_stream = stream;
  h->params.mirror = h->mirror;
  h->mirror_valid = true;
  return NM_OK;
}

// Encodes the I/O tensor maps for (in, out, n) and launches the fused kernel
// on `s`. Arguments are already checked.
nm_status launch_infer(nm_mlp* h, const void* in, int64_t n, void* out, cudaStream_t s) {
  nm_status st = cached_io_maps(h, in, out, n);
  if (st != NM_OK) return st;
  FusedParams& p = h->params;
  p.sched = h->variant == nm::kVarFp8 ? h->sched8 : h->sched;
  p.n = n;
  p.num_tiles = static_cast<int32_t>((n + nm::kTileM - 1) / nm::kTileM);
  p.wait_ns = h->wait_ns;
  p.test_stall = h->test_stall;
  const uint32_t smem = nm::plan_fused_smem(p, h->dims, h->variant, h->smem_optin);
  if (smem == 0) return NM_ERR_UNSUPPORTED;
  if (h->test_check_cols && h->test_check_cols < p.chk_tmem_cols) p.chk_tmem_cols = h->test_check_cols;
  const int grid = p.num_tiles < h->num_sms ? p.num_tiles : h->num_sms;
  const bool after_pack = h->pack_pending && s == h->pack_stream;
  if (nm::launch_fused(p, h->variant, grid, smem, s, !after_pack) != cudaSuccess) return NM_ERR_CUDA;
  if (after_pack) h->pack_pending = false;
  return NM_OK;
}

// Staging buffers of the host-buffer pipeline: freed after the handle's
// streams drain (cudaFree waits for the device anyway).
void free_host_stage(nm_mlp* h) {
  if (!h->hs_stage) return;
  for (int i = 0; i < kHostStreams; ++i)
    if (h->hs[i]) cudaStreamSynchronize(h->hs[i]);
  cudaFree(h->hs_stage);
  h->hs_stage = nullptr;
  h->hs_rows = 0;
}

// Streams, events and staging buffers of nm_mlp_infer_host, created on first
// use. Default chunk: about 12 MiB of input (large enough that the per-chunk
// costs stay small, small enough that filling and draining the pipeline
// stays short), at least 16,384 rows, at most 2^20, a multiple of 128.
nm_status ensure_host_pipeline(nm_mlp* h) {
  if (!h->hs_start) {
    // Each object is created once: after a failure part-way, a later call
    // creates only what is still missing (nm_mlp_destroy frees what exists).
    for (int i = 0; i < kHostStreams; ++i) {
      if (!h->hs[i] && cudaStreamCreateWithFlags(&h->hs[i], cudaStreamNonBlocking) != cudaSuccess) {
        h->hs[i] = nullptr;
        return NM_ERR_CUDA;
      }
      if (!h->hs_done[i] &&
          cudaEventCreateWithFlags(&h->hs_done[i], cudaEventDisableTiming) != cudaSuccess) {
        h->hs_done[i] = nullptr;
        return NM_ERR_CUDA;
      }
    }
    if (cudaEventCreateWithFlags(&h->hs_start, cudaEventDisableTiming) != cudaSuccess) {
      h->hs_start = nullptr;
      return NM_ERR_CUDA;
    }
  }
  if (h->hs_stage) return NM_OK;
  int64_t rows = h->host_chunk;
  if (rows == 0) {
    rows = (static_cast<int64_t>(12) << 20) / (2 * h->dims[0]);
    if (rows < 16384) rows = 16384;
    if (rows > (static_cast<int64_t>(1) << 20)) rows = static_cast<int64_t>(1) << 20;
    rows &= ~static_cast<int64_t>(nm::kTileM - 1);
  }
  const size_t in_bytes = (static_cast<size_t>(rows) * 2u * h->dims[0] + 255u) & ~size_t(255);
  const size_t out_bytes = (static_cast<size_t>(rows) * 2u * h->dims[h->L] + 255u) & ~size_t(255);
  void* p = nullptr;
  if (cudaMalloc(&p, kHostStreams * (in_bytes + out_bytes)) != cudaSuccess) return NM_ERR_OOM;
  h->hs_stage = static_cast<uint8_t*>(p);
  h->hs_rows = rows;
  h->hs_in_bytes = in_bytes;
  h->hs_each = in_bytes + out_bytes;
  return NM_OK;
}

}  // namespace

extern "C" {

int32_t nm_abi_version(void) { return 4; }

const char* nm_status_str(nm_status s) {
  switch (s) {
    case NM_OK: return "NM_OK";
    case NM_ERR_INVALID_ARG: return "NM_ERR_INVALID_ARG";
    case NM_ERR_UNSUPPORTED: return "NM_ERR_UNSUPPORTED";
    case NM_ERR_NOT_PACKED: return "NM_ERR_NOT_PACKED";
    case NM_ERR_OOM: return "NM_ERR_OOM";
    case NM_ERR_CUDA: return "NM_ERR_CUDA";
    case NM_ERR_TIMEOUT: return "NM_ERR_TIMEOUT";
    case NM_ERR_RANGE_CHECK: return "NM_ERR_RANGE_CHECK";
  }
  return "NM_ERR_UNKNOWN";
}

nm_status nm_mlp_plan(const int32_t* dims, int32_t n_dims, nm_variant variant,
                      uint32_t smem_optin, nm_plan* plan) {
  if (!plan) return NM_ERR_INVALID_ARG;
  if (variant != NM_VARIANT_FUSED && variant != NM_VARIANT_ROWMAJOR_WEIGHTS &&
      variant != NM_VARIANT_SCALAR_ACTIVATION && variant != NM_VARIANT_PAIRED_TILES &&
      variant != NM_VARIANT_FP8_WEIGHTS)
    return NM_ERR_INVALID_ARG;
  const nm_status dst = nm::check_dims(dims, n_dims);
  if (dst != NM_OK) return dst;
  const int L = n_dims - 1;
  FusedParams p;
  std::memset(&p, 0, sizeof(p));
  uint32_t w_off[nm::kMaxLayers], rm_off[nm::kMaxLayers], rm_b_off[nm::kMaxLayers];
  size_t mirror_elems = 0;
  nm::net_layout(dims, L, p, w_off, rm_off, rm_b_off, &mirror_elems);
  nm::Schedule* sc = new (std::nothrow) nm::Schedule;
  if (!sc) return NM_ERR_OOM;
  p.sched_bytes = nm::build_schedule(dims, L, w_off, rm_off, *sc, &p.bslab_bytes);
  delete sc;
  const uint32_t smem = nm::plan_fused_smem(p, dims, static_cast<int>(variant), smem_optin);
  if (smem == 0) return NM_ERR_UNSUPPORTED;
  plan->tile_slots = static_cast<int32_t>(p.n_slots);
  plan->warps_per_slot = static_cast<int32_t>(4u * p.n_groups);
  plan->threads = static_cast<int32_t>(p.n_threads);
  plan->streamed_weights = p.stream_w ? 1 : 0;
  plan->weight_stages = p.stream_w ? static_cast<int32_t>(p.n_wstages) : 0;
  plan->input_stages = static_cast<int32_t>(p.n_in_stages);
  plan->output_buffers = static_cast<int32_t>(p.n_out_bufs);
  plan->smem_bytes = smem;
  plan->tmem_columns = p.tmem_cols;
  plan->issuing_warps = p.stream_w ? static_cast<int32_t>(p.n_slots)
                                   : static_cast<int32_t>(p.n_groups_issue);
  plan->a_tmem_k = static_cast<int32_t>(p.a_tmem_k);
  return NM_OK;
}

nm_status nm_mlp_create(const int32_t* dims, int32_t n_dims, nm_mlp** out) {
  if (!out) return NM_ERR_INVALID_ARG;
  *out = nullptr;
  const nm_status dst = nm::check_dims(dims, n_dims);
  if (dst != NM_OK) return dst;
  const int L = n_dims - 1;

  int dev = 0, major = 0, minor = 0, sms = 0, optin = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return NM_ERR_CUDA;
  if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev) != cudaSuccess)
    return NM_ERR_CUDA;
  if (major != 10 || minor != 3) return NM_ERR_UNSUPPORTED;

  nm_mlp* h = new (std::nothrow) nm_mlp();
  if (!h) return NM_ERR_OOM;
  h->L = L;
  h->device = dev;
  h->num_sms = sms;
  h->smem_optin = static_cast<uint32_t>(optin);
  FusedParams& p = h->params;
  std::memset(&p, 0, sizeof(p));
  for (int l = 0; l <= L; ++l) h->dims[l] = dims[l];
  h->blob_size = nm::net_layout(dims, L, p, h->w_off, h->rm_off, h->rm_b_off, &h->mirror_elems);

  nm::Schedule* sc = new (std::nothrow) nm::Schedule;
  if (!sc) {
    delete h;
    return NM_ERR_OOM;
  }
  p.sched_bytes = nm::build_schedule(h->dims, L, h->w_off, h->rm_off, *sc, &p.bslab_bytes);
  nm::set_bias_params(*sc, dims, L, p);
  h->fp8_size = nm::fp8_layout(h->dims, L, h->fp8_off);
  h->fp8_base = h->fp8_size ? nm::align1024(static_cast<uint32_t>(h->blob_size)) : h->blob_size;
  const size_t alloc = h->fp8_base + h->fp8_size;

  if (cudaMalloc(&h->blob, alloc) != cudaSuccess) {
    delete sc;
    delete h;
    return NM_ERR_OOM;
  }
  if (cudaMalloc(&h->status, sizeof(uint32_t)) != cudaSuccess ||
      cudaMalloc(&h->sched, sizeof(nm::Schedule)) != cudaSuccess ||
      (h->fp8_size && cudaMalloc(&h->sched8, sizeof(nm::Schedule)) != cudaSuccess)) {
    cudaFree(h->blob);
    if (h->status) cudaFree(h->status);
    if (h->sched) cudaFree(h->sched);
    delete sc;
    delete h;
    return NM_ERR_OOM;
  }
  bool ok = cudaMemset(h->blob, 0, alloc) == cudaSuccess &&
            cudaMemset(h->status, 0, sizeof(uint32_t)) == cudaSuccess &&
            cudaMemcpy(h->sched, sc, sizeof(nm::Schedule), cudaMemcpyHostToDevice) == cudaSuccess;
  if (ok && h->fp8_size) {
    // Layers 2..L in the FP16-unit view of their E4M3 images.
    for (int l = 1; l < L; ++l) {
      sc->layer[l].K = h->dims[l] >> 1;
      sc->layer[l].w_off = static_cast<uint32_t>(h->fp8_base) + h->fp8_off[l];
    }
    ok = cudaMemcpy(h->sched8, sc, sizeof(nm::Schedule), cudaMemcpyHostToDevice) == cudaSuccess;
  }
  delete sc;
  if (!ok) {
    cudaFree(h->blob);
    cudaFree(h->status);
    cudaFree(h->sched);
    if (h->sched8) cudaFree(h->sched8);
    delete h;
    return NM_ERR_CUDA;
  }
  p.sched = h->sched;
  p.blob = h->blob;
  p.status = h->status;
  *out = h;
  return NM_OK;
}

nm_status nm_mlp_packed_size(const nm_mlp* h, size_t* bytes) {
  if (!h || !bytes) return NM_ERR_INVALID_ARG;
  *bytes = h->blob_size;
  return NM_OK;
}

nm_status nm_mlp_packed_blob(const nm_mlp* h, const void** blob) {
  if (!h || !blob) return NM_ERR_INVALID_ARG;
  *blob = h->blob;
  return NM_OK;
}

nm_status nm_mlp_packed_fp8(const nm_mlp* h, const void** region, size_t* bytes) {
  if (!h || !region || !bytes) return NM_ERR_INVALID_ARG;
  if (!h->fp8_size) return NM_ERR_UNSUPPORTED;
  if (!h->packed || !h->fp8_valid) return NM_ERR_NOT_PACKED;
  *region = h->blob + h->fp8_base;
  *bytes = h->fp8_size;
  return NM_OK;
}

nm_status nm_mlp_pack_weights(nm_mlp* h, const void* const* W, const void* const* b,
                              nm_stream stream) {
  if (!h || !W || !b) return NM_ERR_INVALID_ARG;
  PackParams pp = make_pack_params(h);
  for (int l = 0; l < h->L; ++l) {
    if (!W[l] || !b[l] || !aligned16(W[l]) || !aligned16(b[l])) return NM_ERR_INVALID_ARG;
    pp.rm_w[l] = const_cast<uint16_t*>(static_cast<const uint16_t*>(W[l]));
    pp.rm_b[l] = const_cast<uint16_t*>(static_cast<const uint16_t*>(b[l]));
  }
  if (nm::launch_pack(pp, false, h->num_sms, reinterpret_cast<cudaStream_t>(stream)) != cudaSuccess)
    return NM_ERR_CUDA;
  h->fp8_valid = false;
  if (h->variant == nm::kVarFp8) {
    // part of the pack the caller asked for: captured with it if it is
    const nm_status st = ensure_fp8(h, reinterpret_cast<cudaStream_t>(stream), true);
    if (st != NM_OK) return st;
  }
  h->packed = true;
  h->mirror_valid = false;
  h->pack_pending = true;
  h->pack_stream = reinterpret_cast<cudaStream_t>(stream);
  return NM_OK;
}

nm_status nm_mlp_unpack_weights(const nm_mlp* h, void* const* W, void* const* b, nm_stream stream) {
  if (!h || !W || !b) return NM_ERR_INVALID_ARG;
  if (!h->packed) return NM_ERR_NOT_PACKED;
  PackParams pp = make_pack_params(h);
  for (int l = 0; l < h->L; ++l) {
    if (!W[l] || !b[l] || !aligned16(W[l]) || !aligned16(b[l])) return NM_ERR_INVALID_ARG;
    pp.rm_w[l] = static_cast<uint16_t*>(W[l]);
    pp.rm_b[l] = static_cast<uint16_t*>(b[l]);
  }
  if (nm::launch_pack(pp, true, h->num_sms, reinterpret_cast<cudaStream_t>(stream)) != cudaSuccess)
    return NM_ERR_CUDA;
  return NM_OK;
}

nm_status nm_mlp_infer(nm_mlp* h, const void* in, int64_t n, void* out, nm_stream stream) {
  if (!h) return NM_ERR_INVALID_ARG;
  if (n < 0 || n > kMaxRows) return NM_ERR_INVALID_ARG;
  if (n == 0) return NM_OK;
  if (!in || !out || !aligned16(in) || !aligned16(out)) return NM_ERR_INVALID_ARG;
  if (!h->packed) return NM_ERR_NOT_PACKED;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  if (h->variant == nm::kVarRowMajor) {
    const nm_status st = ensure_mirror(h, s);
    if (st != NM_OK) return st;
  }
  if (h->variant == nm::kVarFp8) {
    const nm_status st = ensure_fp8(h, s);
    if (st != NM_OK) return st;
  }
  return launch_infer(h, in, n, out, s);
}

nm_status nm_mlp_infer_host(nm_mlp* h, const void* host_in, int64_t n, void* host_out,
                            nm_stream stream) {
  if (!h) return NM_ERR_INVALID_ARG;
  if (n < 0 || n > kMaxRows) return NM_ERR_INVALID_ARG;
  if (n == 0) return NM_OK;
  if (!host_in || !host_out) return NM_ERR_INVALID_ARG;
  if (!h->packed) return NM_ERR_NOT_PACKED;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  if (h->variant == nm::kVarRowMajor) {
    const nm_status st = ensure_mirror(h, s);
    if (st != NM_OK) return st;
  }
  if (h->variant == nm::kVarFp8) {
    const nm_status st = ensure_fp8(h, s);
    if (st != NM_OK) return st;
  }
  nm_status st = ensure_host_pipeline(h);
  if (st != NM_OK) return st;
  const size_t in_row = 2u * static_cast<size_t>(h->dims[0]);
  const size_t out_row = 2u * static_cast<size_t>(h->dims[h->L]);
  // The handle's streams start after the caller's prior work ...
  if (cudaEventRecord(h->hs_start, s) != cudaSuccess) return NM_ERR_CUDA;
  for (int i = 0; i < kHostStreams; ++i)
    if (cudaStreamWaitEvent(h->hs[i], h->hs_start, 0) != cudaSuccess) return NM_ERR_CUDA;
  // ... run the chunks: copy in, evaluate, copy out, each chunk in order on
  // its stream, so neighbouring chunks overlap ...
  int i = 0;
  for (int64_t r0 = 0; r0 < n; r0 += h->hs_rows, i = (i + 1) % kHostStreams) {
    const int64_t m = (n - r0 < h->hs_rows) ? (n - r0) : h->hs_rows;
    uint8_t* din = h->hs_stage + static_cast<size_t>(i) * h->hs_each;
    uint8_t* dout = din + h->hs_in_bytes;
    const uint8_t* src = static_cast<const uint8_t*>(host_in) + static_cast<size_t>(r0) * in_row;
    uint8_t* dst = static_cast<uint8_t*>(host_out) + static_cast<size_t>(r0) * out_row;
    if (cudaMemcpyAsync(din, src, static_cast<size_t>(m) * in_row, cudaMemcpyHostToDevice,
                        h->hs[i]) != cudaSuccess)
      return NM_ERR_CUDA;
    if ((st = launch_infer(h, din, m, dout, h->hs[i])) != NM_OK) return st;
    if (cudaMemcpyAsync(dst, dout, static_cast<size_t>(m) * out_row, cudaMemcpyDeviceToHost,
                        h->hs[i]) != cudaSuccess)
      return NM_ERR_CUDA;
  }
  // ... and the caller's stream waits for all of them.
  for (int k = 0; k < kHostStreams; ++k) {
    if (cudaEventRecord(h->hs_done[k], h->hs[k]) != cudaSuccess) return NM_ERR_CUDA;
    if (cudaStreamWaitEvent(s, h->hs_done[k], 0) != cudaSuccess) return NM_ERR_CUDA;
  }
  return NM_OK;
}

nm_status nm_mlp_set_host_chunk(nm_mlp* h, int64_t rows) {
  if (!h) return NM_ERR_INVALID_ARG;
  if (rows != 0 && (rows < nm::kTileM || rows > (static_cast<int64_t>(1) << 20) || rows % nm::kTileM))
    return NM_ERR_INVALID_ARG;
  if (rows == h->host_chunk) return NM_OK;
  h->host_chunk = rows;
  free_host_stage(h);
  return NM_OK;
}

nm_status nm_mlp_set_variant(nm_mlp* h, nm_variant v) {
  if (!h) return NM_ERR_INVALID_ARG;
  if (v != NM_VARIANT_FUSED && v != NM_VARIANT_ROWMAJOR_WEIGHTS && v != NM_VARIANT_SCALAR_ACTIVATION &&
      v != NM_VARIANT_PAIRED_TILES && v != NM_VARIANT_FP8_WEIGHTS)
    return NM_ERR_INVALID_ARG;
  if (v == NM_VARIANT_FP8_WEIGHTS && !h->fp8_size) return NM_ERR_UNSUPPORTED;
  h->variant = static_cast<int>(v);
  return NM_OK;
}

nm_status nm_mlp_device_status(nm_mlp* h, nm_stream stream) {
  if (!h) return NM_ERR_INVALID_ARG;
  if (cudaStreamSynchronize(reinterpret_cast<cudaStream_t>(stream)) != cudaSuccess) return NM_ERR_CUDA;
  uint32_t v = 0;
  if (cudaMemcpy(&v, h->status, sizeof(v), cudaMemcpyDeviceToHost) != cudaSuccess) return NM_ERR_CUDA;
  if (v != 0) {
    if (cudaMemset(h->status, 0, sizeof(uint32_t)) != cudaSuccess) return NM_ERR_CUDA;
    return (v & nm::kStatusRangeCheck) ? NM_ERR_RANGE_CHECK : NM_ERR_TIMEOUT;
  }
  return NM_OK;
}

nm_status nm_mlp_set_wait_limit(nm_mlp* h, uint64_t nanoseconds) {
  if (!h) return NM_ERR_INVALID_ARG;
  h->wait_ns = nanoseconds;
  return NM_OK;
}

nm_status nm_mlp_set_test_stall(nm_mlp* h, int32_t enable) {
  if (!h) return NM_ERR_INVALID_ARG;
  h->test_stall = enable ? 1u : 0u;
  return NM_OK;
}

nm_status nm_mlp_set_test_check_limit(nm_mlp* h, uint32_t tmem_columns) {
  if (!h) return NM_ERR_INVALID_ARG;
  h->test_check_cols = tmem_columns;
  return NM_OK;
}

int32_t nm_checking_build(void) {
#ifdef NM_RANGE_CHECKS
  return 1;
#else
  return 0;
#endif
}

void nm_mlp_destroy(nm_mlp* h) {
  if (!h) return;
  cudaDeviceSynchronize();
  free_host_stage(h);
  for (int i = 0; i < kHostStreams; ++i) {
    if (h->hs[i]) cudaStreamDestroy(h->hs[i]);
    if (h->hs_done[i]) cudaEventDestroy(h->hs_done[i]);
  }
  if (h->hs_start) cudaEventDestroy(h->hs_start);
  cudaFree(h->blob);
  cudaFree(h->status);
  cudaFree(h->sched);
  if (h->sched8) cudaFree(h->sched8);
  if (h->mirror) cudaFree(h->mirror);
  delete h;
}

}  // extern "C"
