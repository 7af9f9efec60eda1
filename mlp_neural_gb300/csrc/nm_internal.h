// nm_internal.h -- declarations shared by the translation units of libnmmlp
// (kernel parameter blocks and launchers). Not part of the public ABI.
#pragma once

#include <cstdint>
#include <cuda.h>
#include <cuda_runtime.h>

#include "nm_layout.cuh"

namespace nm {

constexpr int kSlots = 2;          // 128-sample tiles in flight per CTA
constexpr int kMaxInStages = 4;    // input TMA ring depth (upper bound)
constexpr int kMaxBStages = 4;     // B-operand ring depth of the row-major ablation
constexpr int kFusedThreads = 192; // warp 0 producer, warp 1 MMA, warps 2-5 epilogue
constexpr uint32_t kStatusTimeout = 1u;

enum Variant : int { kVarFused = 0, kVarRowMajor = 1, kVarScalar = 2 };

// Barrier slots inside the barrier block of the fused kernel's smem.
enum BarIndex : int {
  kBarInFull = 0,
  kBarInEmpty = kBarInFull + kMaxInStages,
  kBarAccFull = kBarInEmpty + kMaxInStages,
  kBarActReady = kBarAccFull + kSlots,
  kBarBFull = kBarActReady + kSlots,
  kBarBEmpty = kBarBFull + kMaxBStages,
  kBarWLoad = kBarBEmpty + kMaxBStages,
  kBarDrain = kBarWLoad + 1,
  kBarNever = kBarDrain + 1,  // never signalled (failure-path test hook)
  kBarCount = kBarNever + 1
};
constexpr uint32_t kBarBlockBytes = 256;  // kBarCount * 8 barriers, then TMEM address and abort flag
constexpr uint32_t kTmemSlotOff = 192;
constexpr uint32_t kAbortOff = 196;
static_assert(kBarCount * 8 <= kTmemSlotOff, "barrier block overflow");

struct FusedParams {  // 128-byte aligned through its CUtensorMap members
  CUtensorMap tm_in[3];   // input [n][d0] maps, by swizzle kind (box 128 rows)
  CUtensorMap tm_out[3];  // output [n][dL] maps, by swizzle kind (box 32 rows)
  const uint8_t* blob;    // packed weight images + FP16 biases
  const uint16_t* mirror; // row-major weights (row-major ablation only)
  uint32_t* status;       // device status word
  int64_t n;
  int32_t num_tiles;
  int32_t L;
  int32_t dims[kMaxLayers + 1];
  uint32_t w_off[kMaxLayers];       // byte offset of layer l's image in blob / smem weight region
  uint32_t rm_off[kMaxLayers];      // element offset of W_l in the mirror
  uint32_t bias_f_off[kMaxLayers];  // float offset of b_l in the smem bias array
  uint32_t bias_off;                // byte offset of the bias block in the blob
  uint32_t n_bias;                  // sum of d_1..d_L
  // shared-memory plan (byte offsets from the 1024-aligned base)
  uint32_t sm_w, sm_bias, sm_in, sm_act, sm_out, sm_b, sm_bar;
  uint32_t in_stage_bytes, act_slot_bytes, out_slot_bytes, b_stage_bytes;
  uint32_t n_in_stages, n_b_stages;
  uint32_t tmem_cols;  // allocated TMEM columns (power of two)
  uint32_t nmax;       // TMEM columns per tile slot (max layer width)
  uint64_t wait_ns;    // limit of every pipeline wait
  uint32_t test_stall; // non-zero: the MMA thread first waits on kBarNever
};

// Returns the dynamic smem bytes the plan needs, or 0 if it does not fit.
uint32_t plan_fused_smem(FusedParams& p, int variant, uint32_t smem_optin);

cudaError_t launch_fused(const FusedParams& p, int variant, int grid, uint32_t smem,
                         cudaStream_t stream);

struct PackParams {
  int32_t L;
  int32_t dims[kMaxLayers + 1];
  uint32_t w_off[kMaxLayers];
  uint32_t bias_off;
  uint32_t chunk_start[kMaxLayers + 1];  // first 16-byte weight chunk of each layer
  uint32_t bias_chunk_start[kMaxLayers + 1];
  uint16_t* rm_w[kMaxLayers];  // row-major weights (source of pack, destination of unpack)
  uint16_t* rm_b[kMaxLayers];
  uint8_t* blob;
};

cudaError_t launch_pack(const PackParams& p, bool unpack, int num_sms, cudaStream_t stream);

}  // namespace nm
