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

// Once per device, with that device current: the scratch array's device
// address, the device's SM count and shared-memory limit. Returns NM_OK or
// the failing status.
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
    d.scratch = static_cast<uint8_t*>(ptr);
    d.num_sms = sms;
    d.smem_optin = static_cast<uint32_t>(optin);
    d.ready = true;
  }
  out = d;
  return NM_OK;
}

}  // namespace

extern "C" nm_status nm_mlp_infer_noalloc(const int32_t* dims, int32_t n_dims,
                                          const void* const* W, const void* const* b,
                                          const void* in, int64_t n, void* out,
                                          nm_stream stream) {
  // ---- arguments (all checked before any device work)
  if (!W || !b) return NM_ERR_INVALID_ARG;
  nm_status st = nm::check_dims(dims, n_dims);
  if (st != NM_OK) return st;
  const int L = n_dims - 1;
  for (int l = 0; l < L; ++l)
    if (!W[l] || !b[l] || !nm::aligned16(W[l]) || !nm::aligned16(b[l])) return NM_ERR_INVALID_ARG;
  if (n < 0 || n > nm::kMaxRows) return NM_ERR_INVALID_ARG;
  if (n == 0) return NM_OK;
  if (!in || !out || !nm::aligned16(in) || !nm::aligned16(out)) return NM_ERR_INVALID_ARG;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  // The call ends by synchronising `stream`, which a stream being captured
  // into a graph does not allow: refuse before enqueuing anything.
  cudaStreamCaptureStatus cap = cudaStreamCaptureStatusNone;
  if (cudaStreamIsCapturing(s, &cap) != cudaSuccess) return NM_ERR_CUDA;
  if (cap != cudaStreamCaptureStatusNone) return NM_ERR_UNSUPPORTED;

  // ---- layout of the packed weights (the definition nm_mlp_create uses)
  nm::FusedParams p;
  std::memset(&p, 0, sizeof(p));
  uint32_t w_off[nm::kMaxLayers] = {}, rm_off[nm::kMaxLayers] = {};
  const size_t blob_size = nm::net_layout(dims, L, p, w_off, rm_off, nullptr, nullptr);
  if (kBlobOff + blob_size > kNoAllocScratchBytes) return NM_ERR_UNSUPPORTED;  // exceeds the scratch

  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return NM_ERR_CUDA;
  if (dev < 0 || dev >= kMaxDevices) return NM_ERR_UNSUPPORTED;
  DeviceSetup ds;
  st = setup_device(dev, ds);
  if (st != NM_OK) return st;
  uint8_t* status = ds.scratch + kStatusOff;
  uint8_t* sched = ds.scratch + kSchedOff;
  uint8_t* blob = ds.scratch + kBlobOff;

  // ---- schedule table and parameters (host stack only)
  nm::Schedule sc;
  p.sched_bytes = nm::build_schedule(dims, L, w_off, rm_off, sc, &p.bslab_bytes);
  nm::set_bias_params(sc, dims, L, p);
  p.blob = blob;
  p.sched = sched;
  p.status = reinterpret_cast<uint32_t*>(status);
  p.n = n;
  p.num_tiles = static_cast<int32_t>((n + nm::kTileM - 1) / nm::kTileM);
  p.wait_ns = 2000000000ull;
  const uint32_t smem = nm::plan_fused_smem(p, dims, nm::kVarFused, ds.smem_optin);
  if (smem == 0) return NM_ERR_UNSUPPORTED;
  if ((st = nm::encode_io_maps(p, dims, L, in, out, n)) != NM_OK) return st;

  // ---- device work, all on `stream`. The scratch keeps the previous call's
  // contents: the status word and the blob (whose padding must be zero) are
  // cleared first.
  if (cudaMemsetAsync(status, 0, sizeof(uint32_t), s) != cudaSuccess ||
      cudaMemsetAsync(blob, 0, blob_size, s) != cudaSuccess ||
      cudaMemcpyAsync(sched, &sc, p.sched_bytes, cudaMemcpyHostToDevice, s) != cudaSuccess)
    return NM_ERR_CUDA;
  nm::PackParams pp = nm::make_pack_params(dims, L, w_off, p.bias_off, blob);
  for (int l = 0; l < L; ++l) {
    pp.rm_w[l] = const_cast<uint16_t*>(static_cast<const uint16_t*>(W[l]));
    pp.rm_b[l] = const_cast<uint16_t*>(static_cast<const uint16_t*>(b[l]));
  }
  if (nm::launch_pack(pp, false, ds.num_sms, s) != cudaSuccess) return NM_ERR_CUDA;
  const int grid = p.num_tiles < ds.num_sms ? p.num_tiles : ds.num_sms;
  if (nm::launch_fused(p, nm::kVarFused, grid, smem, s, false) != cudaSuccess) return NM_ERR_CUDA;

  // ---- completion: this entry point returns only once `stream` has run the
  // work, so that a kernel-side give-up can be reported.
  if (cudaStreamSynchronize(s) != cudaSuccess) return NM_ERR_CUDA;
  uint32_t word = 0;
  if (cudaMemcpy(&word, status, sizeof(word), cudaMemcpyDeviceToHost) != cudaSuccess)
    return NM_ERR_CUDA;
  if (word & nm::kStatusRangeCheck) return NM_ERR_RANGE_CHECK;
  return word ? NM_ERR_TIMEOUT : NM_OK;
}
