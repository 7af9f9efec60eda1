// nm_noalloc.cu -- inference for callers that must not allocate device memory.
//
// Some callers cannot call cudaMalloc: code that runs inside a host
// application which owns the whole device memory budget (a renderer or a
// game engine with its own pool), or a latency-critical path where an
// allocation's implicit synchronisation is not allowed. They can still hand
// over device buffers they already own. nm_mlp_infer_noalloc serves them: it
// takes the network's row-major weights, the inputs and the outputs from the
// caller, and keeps everything else it needs (the packed weights, the
// schedule table and the status word) in one file-scope device array,
// g_noalloc_scratch, of kNoAllocScratchBytes. That array is part of the
// library's module: every GPU that loads the library holds it until the
// process exits.
//
// In host code the array's name is only a host-side stand-in, not a device
// address. The device address is obtained here, once per device, with that
// device current, by cudaGetSymbolAddress, and passed to the kernels.
#include <cuda.h>
#include <cuda_runtime.h>
#include <cudaTypedefs.h>

#include <cstdint>
#include <cstring>
#include <mutex>

#include "nm_internal.h"
#include "nm_mlp.h"

namespace {

constexpr size_t kNoAllocScratchBytes = size_t(1) << 20;  // 1 MiB
constexpr size_t kStatusOff = 0;                          // 4-byte status word
constexpr size_t kSchedOff = 256;                         // nm::Schedule
constexpr size_t kBlobOff = (kSchedOff + sizeof(nm::Schedule) + 1023) & ~size_t(1023);
static_assert(kBlobOff < kNoAllocScratchBytes, "scratch layout");

static __device__ __align__(256) uint8_t g_noalloc_scratch[kNoAllocScratchBytes];

constexpr int kMaxDevices = 64;

struct DeviceSetup {
  bool ready = false;
  uint8_t* scratch = nullptr;  // device address of g_noalloc_scratch on this device
  int num_sms = 0;
  uint32_t smem_optin = 0;
};

std::mutex g_setup_mu;
DeviceSetup g_setup[kMaxDevices];
PFN_cuTensorMapEncodeTiled_v12000 g_encode_na = nullptr;

// Once per device, with that device current: the scratch array's device
// address, the device's SM count and shared-memory limit, and the tensor-map
// encoder. Returns NM_OK or the failing status.
nm_status setup_device(int dev, DeviceSetup& out) {
  std::lock_guard<std::mutex> lk(g_setup_mu);
  DeviceSetup& d = g_setup[dev];
  if (!d.ready) {
    int major = 0, minor = 0, sms = 0, optin = 0;
    if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev) != cudaSuccess)
      return NM_ERR_CUDA;
    if (major != 10 || minor != 3) return NM_ERR_UNSUPPORTED;
    void* ptr = nullptr;
    if (cudaGetSymbolAddress(&ptr, g_noalloc_scratch) != cudaSuccess || ptr == nullptr)
      return NM_ERR_CUDA;
    if (!g_encode_na) {
      void* fn = nullptr;
      cudaDriverEntryPointQueryResult q;
      if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault,
                                           &q) != cudaSuccess ||
          q != cudaDriverEntryPointSuccess)
        return NM_ERR_CUDA;
      g_encode_na = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
    }
    d.scratch = static_cast<uint8_t*>(ptr);
    d.num_sms = sms;
    d.smem_optin = static_cast<uint32_t>(optin);
    d.ready = true;
  }
  out = d;
  return NM_OK;
}

nm_status encode(CUtensorMap* m, const void* ptr, int width, int64_t rows, int box_w, int box_rows) {
  cuuint64_t gdim[2] = {static_cast<cuuint64_t>(width), static_cast<cuuint64_t>(rows)};
  cuuint64_t gstride[1] = {static_cast<cuuint64_t>(width) * 2u};
  cuuint32_t box[2] = {static_cast<cuuint32_t>(box_w), static_cast<cuuint32_t>(box_rows)};
  cuuint32_t estride[2] = {1, 1};
  const CUtensorMapSwizzle sw = box_w == 64 ? CU_TENSOR_MAP_SWIZZLE_128B
                                : box_w == 32 ? CU_TENSOR_MAP_SWIZZLE_64B
                                              : CU_TENSOR_MAP_SWIZZLE_32B;
  const CUresult r = g_encode_na(m, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 2, const_cast<void*>(ptr),
                                 gdim, gstride, box, estride, CU_TENSOR_MAP_INTERLEAVE_NONE, sw,
                                 CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                                 CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? NM_OK : NM_ERR_CUDA;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

}  // namespace

extern "C" nm_status nm_mlp_infer_noalloc(const int32_t* dims, int32_t n_dims,
                                          const void* const* W, const void* const* b,
                                          const void* in, int64_t n, void* out,
                                          nm_stream stream) {
  // ---- arguments (all checked before any device work)
  if (!dims || n_dims < 2 || !W || !b) return NM_ERR_INVALID_ARG;
  const int L = n_dims - 1;
  if (L > nm::kMaxLayers) return NM_ERR_UNSUPPORTED;
  for (int l = 0; l <= L; ++l)
    if (dims[l] < 16 || dims[l] > nm::kMaxDim || dims[l] % 16 != 0) return NM_ERR_UNSUPPORTED;
  for (int l = 0; l < L; ++l)
    if (!W[l] || !b[l] || !aligned16(W[l]) || !aligned16(b[l])) return NM_ERR_INVALID_ARG;
  if (n < 0 || n > (static_cast<int64_t>(1) << 31) - 128) return NM_ERR_INVALID_ARG;
  if (n == 0) return NM_OK;
  if (!in || !out || !aligned16(in) || !aligned16(out)) return NM_ERR_INVALID_ARG;

  // ---- layout of the packed weights (same definition as nm_mlp_create)
  uint32_t w_off[nm::kMaxLayers] = {}, rm_off[nm::kMaxLayers] = {};
  uint32_t off = 0, nb = 0;
  for (int l = 0; l < L; ++l) {
    off = nm::align1024(off);
    w_off[l] = off;
    off += nm::image_bytes(static_cast<uint32_t>(dims[l + 1]), dims[l]);
    nb += static_cast<uint32_t>(dims[l + 1]);
  }
  const uint32_t bias_off = nm::align1024(off);
  const size_t blob_size = bias_off + 2u * nb;
  if (kBlobOff + blob_size > kNoAllocScratchBytes) return NM_ERR_UNSUPPORTED;  // exceeds the scratch

  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return NM_ERR_CUDA;
  if (dev < 0 || dev >= kMaxDevices) return NM_ERR_UNSUPPORTED;
  DeviceSetup ds;
  nm_status st = setup_device(dev, ds);
  if (st != NM_OK) return st;
  uint8_t* status = ds.scratch + kStatusOff;
  uint8_t* sched = ds.scratch + kSchedOff;
  uint8_t* blob = ds.scratch + kBlobOff;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);

  // ---- schedule table and parameters (host stack only)
  nm::Schedule sc;
  nm::FusedParams p;
  std::memset(&p, 0, sizeof(p));
  p.L = L;
  p.bias_off = bias_off;
  p.sched_bytes = nm::build_schedule(dims, L, w_off, rm_off, sc, &p.bslab_bytes);
  {
    uint32_t row0 = 0;
    for (int l = 0; l < L; ++l) {
      p.bias_row0[l] = row0;
      p.bslab_off[l] = sc.layer[l].bslab_off;
      row0 += static_cast<uint32_t>(dims[l + 1]);
    }
    p.n_bias = row0;
  }
  p.blob = blob;
  p.sched = sched;
  p.status = reinterpret_cast<uint32_t*>(status);
  p.n = n;
  p.num_tiles = static_cast<int32_t>((n + nm::kTileM - 1) / nm::kTileM);
  p.wait_ns = 2000000000ull;
  const uint32_t smem = nm::plan_fused_smem(p, dims, nm::kVarFused, ds.smem_optin);
  if (smem == 0) return NM_ERR_UNSUPPORTED;

  int w[16], k0[16];
  int ns = nm::segments(dims[0], w, k0);
  for (int i = 0; i < ns; ++i)
    if ((st = encode(&p.tm_in[nm::swizzle_kind(w[i])], in, dims[0], n, w[i], nm::kTileM)) != NM_OK)
      return st;
  if (dims[L] >= 32 &&
      (st = encode(&p.tm_out[nm::swizzle_kind(32)], out, dims[L], n, 32, 32)) != NM_OK)
    return st;
  if ((dims[L] & 31) &&
      (st = encode(&p.tm_out[nm::swizzle_kind(16)], out, dims[L], n, 16, 32)) != NM_OK)
    return st;

  // ---- device work, all on `stream`. The scratch keeps the previous call's
  // contents: the status word and the blob (whose padding must be zero) are
  // cleared first.
  if (cudaMemsetAsync(status, 0, sizeof(uint32_t), s) != cudaSuccess ||
      cudaMemsetAsync(blob, 0, blob_size, s) != cudaSuccess ||
      cudaMemcpyAsync(sched, &sc, p.sched_bytes, cudaMemcpyHostToDevice, s) != cudaSuccess)
    return NM_ERR_CUDA;
  nm::PackParams pp;
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
    pp.rm_w[l] = const_cast<uint16_t*>(static_cast<const uint16_t*>(W[l]));
    pp.rm_b[l] = const_cast<uint16_t*>(static_cast<const uint16_t*>(b[l]));
  }
  pp.chunk_start[L] = cw;
  pp.bias_chunk_start[L] = cb;
  pp.bias_off = bias_off;
  pp.blob = blob;
  if (nm::launch_pack(pp, false, ds.num_sms, s) != cudaSuccess) return NM_ERR_CUDA;
  const int grid = p.num_tiles < ds.num_sms ? p.num_tiles : ds.num_sms;
  if (nm::launch_fused(p, nm::kVarFused, grid, smem, s, false) != cudaSuccess) return NM_ERR_CUDA;

  // ---- completion: this entry point returns only once `stream` has run the
  // work, so that a kernel-side give-up can be reported.
  if (cudaStreamSynchronize(s) != cudaSuccess) return NM_ERR_CUDA;
  uint32_t word = 0;
  if (cudaMemcpy(&word, status, sizeof(word), cudaMemcpyDeviceToHost) != cudaSuccess)
    return NM_ERR_CUDA;
  return word ? NM_ERR_TIMEOUT : NM_OK;
}
