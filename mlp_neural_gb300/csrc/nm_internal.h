// nm_internal.h -- declarations shared by the translation units of libnmmlp
// (kernel parameter blocks, the per-network schedule table, launchers).
// Not part of the public ABI.
#pragma once

#include <cstdint>
#include <cuda.h>
#include <cuda_runtime.h>

#include "nm_layout.cuh"
#include "nm_mlp.h"

namespace nm {

constexpr int kMaxSlots = 5;       // 128-sample tiles in flight per CTA (upper bound)
constexpr int kMaxInStages = 2 * kMaxSlots;  // input TMA ring: up to 2 stages per slot
constexpr int kMaxBStages = kMaxSlots;       // row-major ablation: one B stage per slot
// Resident weights: warps 0 .. S-1 issue the slots' MMA chains (one warp per
// tile slot), warp S produces the input tiles, and from warp kEpiWarp0 on
// each slot has 4G epilogue warps (4 TMEM lane quadrants x G column groups);
// warps between the producer and kEpiWarp0 have no role.
constexpr int kEpiWarp0 = 8;
constexpr int kMaxEpiWarps = 4 * kMaxSlots > 16 ? 4 * kMaxSlots : 16;
constexpr int kMaxResidentWarps = kEpiWarp0 + kMaxEpiWarps;
// Streamed weights: the slots' warps (at most 16: 1 slot x 16, 2 x 8 or
// 3 x 4), one weight-producer warp and one input-producer warp.
constexpr int kStreamSlots = 3;    // tile slots at most with streamed weights
constexpr int kOutBufs = 2;        // output staging buffers per slot (TMA-store double buffer)
constexpr int kMaxSlabs = kMaxLayers * (kMaxDim / 16);
constexpr uint32_t kStatusTimeout = 1u;
// Set by the checking build (NM_RANGE_CHECKS) when an address the kernel is
// about to use falls outside the plan's tensor or shared memory.
constexpr uint32_t kStatusRangeCheck = 2u;

// Public variants 0..4 (nm_variant); 8 and 9 are the fused and the
// scalar-activation kernels with streamed instead of resident weights, chosen
// by the planner when the packed weights do not fit in shared memory; 11 is
// the fused streamed kernel for plans that keep part of A in shared memory
// (its own instantiation, so the other streamed plans run code without those
// branches); 10 is the narrow-precision variant, which always streams its
// weights. The paired-tiles variant runs the fused kernel with a plan that
// issues the tile regions two at a time.
enum Variant : int {
  kVarFused = 0,
  kVarRowMajor = 1,
  kVarScalar = 2,
  kVarPaired = 3,
  kVarFp8 = 4,
  kVarFusedStream = 8,
  kVarScalarStream = 9,
  kVarFp8Stream = 10,
  kVarFusedStreamSplitA = 11
};
constexpr int kMaxWStages = 4;     // streamed-weight ring depth (upper bound)

// Barrier slots inside the barrier block of the fused kernel's smem. Input
// stage s * n_in_stages + k belongs to slot s; the row-major ablation's B
// stage s belongs to slot s.
enum BarIndex : int {
  kBarInFull = 0,
  kBarInEmpty = kBarInFull + kMaxInStages,
  kBarAccFull = kBarInEmpty + kMaxInStages,
  kBarBEmpty = kBarAccFull + kMaxSlots,
  kBarWFull = kBarBEmpty + kMaxBStages,   // streamed-weight ring
  kBarWEmpty = kBarWFull + kMaxWStages,
  kBarWLoad = kBarWEmpty + kMaxWStages,
  kBarDrain = kBarWLoad + 1,  // one per slot
  kBarNever = kBarDrain + kMaxSlots,  // never signalled (failure-path test hook)
  kBarCount = kBarNever + 1
};
constexpr uint32_t kTmemSlotOff = 512;  // barriers first, then the TMEM address and abort flag
constexpr uint32_t kAbortOff = 516;
static_assert(kBarCount * 8 <= kTmemSlotOff, "barrier block overflow");

// Per-layer schedule entry (host-built, copied to smem once per CTA).
struct LayerInfo {
  int32_t K, N;
  uint32_t slab_begin, slab_end;  // range of this layer's k-slabs in the descriptor table
  uint32_t idesc;                 // tcgen05 instruction descriptor (M = 128, N)
  uint32_t bslab_off;             // byte offset of b_l's bias slab in the bias-slab region
  uint32_t rm_off;                // element offset of W_l in the row-major mirror
  uint32_t w_off;                 // byte offset of W_l's image in the blob / smem weight region
};

// UMMA shared-memory descriptors of one 16-wide k-slab, with start addresses
// relative to a base that the kernel adds at issue time: A relative to the
// layer's A tile, B relative to the layer's B image (resident weights or the
// row-major ablation's B stage).
struct SlabDesc {
  uint64_t a;
  uint64_t b;
};

struct Schedule {
  LayerInfo layer[kMaxLayers];
  SlabDesc slab[kMaxSlabs];
};
static_assert(sizeof(LayerInfo) == 32, "layer table entry size");
static_assert(sizeof(Schedule) % 16 == 0, "schedule must copy in 16-byte units");

// Fills the schedule for a network and returns the number of bytes of it the
// kernel copies to shared memory (layer table + the slabs in use); *bslab_bytes
// receives the size of the bias-slab region.
uint32_t build_schedule(const int32_t* dims, int L, const uint32_t* w_off, const uint32_t* rm_off,
                        Schedule& s, uint32_t* bslab_bytes);

// The bias enters through the tensor core: every layer's MMA chain ends with
// one more K=16 MMA whose A slab is a "ones" column (A[r][0] = 1, the rest 0)
// in shared memory and whose B slab is the "bias slab" (B[n][0] = b[n], the
// rest 0), both in the 32-byte-swizzle K-major layout. It adds b[n] to the
// FP32 accumulator after the sum of products, as the arithmetic prescribes.
constexpr uint32_t kOnesTileBytes = 128u * 32u;

struct FusedParams {  // 128-byte aligned through its CUtensorMap members
  CUtensorMap tm_in[3];   // input [n][d0] maps, by swizzle kind (box 128 rows)
  CUtensorMap tm_out[3];  // output [n][dL] maps, by swizzle kind (box 32 rows)
  const uint8_t* blob;    // packed weight images + FP16 biases
  const uint8_t* sched;   // Schedule (device copy)
  const uint16_t* mirror; // row-major weights (row-major ablation only)
  uint32_t* status;       // device status word
  int64_t n;
  int32_t num_tiles;
  int32_t L;
  int32_t d0, dL;
  uint32_t bias_off;      // byte offset of the bias block in the blob (= weight image bytes)
  uint32_t n_bias;        // sum of d_1..d_L
  uint32_t sched_bytes;   // bytes of the schedule to copy
  uint32_t bslab_bytes;   // bytes of the bias-slab region
  uint64_t nslab_bits;    // 4 bits per layer: K_l / 16 - 1
  uint64_t n16_bits;      // 4 bits per layer: N_l / 16 - 1
  uint32_t bias_row0[kMaxLayers];  // index of b_l[0] among the concatenated biases
  uint32_t bslab_off[kMaxLayers];  // byte offset of b_l's slab in the bias-slab region
  // shared-memory plan (byte offsets from the 1024-aligned base)
  uint32_t sm_w, sm_sched, sm_bslab, sm_ones, sm_in, sm_out, sm_b, sm_wring, sm_bar;
  uint32_t in_stage_bytes, out_slot_bytes, b_stage_bytes;
  uint32_t n_in_stages;  // input stages per slot
  uint32_t n_b_stages, n_out_bufs;
  uint32_t n_slots;     // tiles in flight (tile regions of TMEM)
  // Resident weights: the tile regions are issued in groups of one or two
  // regions, one issuing warp and one named barrier per group; group g
  // covers regions grp_first[g] .. grp_first[g] + grp_tiles[g] - 1.
  uint32_t n_groups_issue;
  uint32_t grp_first[kMaxSlots], grp_tiles[kMaxSlots], grp_of[kMaxSlots];
  uint32_t n_groups;    // column groups of a slot's epilogue (4 * n_groups warps per slot)
  uint32_t n_threads;   // block size
  uint32_t tmem_cols;   // allocated TMEM columns (power of two)
  uint32_t slot_cols;   // TMEM columns per tile slot
  // Resident weights: a slot holds its accumulator (columns [0, a_col)) and
  // the next layer's FP16 A (from a_col); one "ones" slab (8 columns) at
  // ones_col serves every slot's bias MMA.
  uint32_t a_col, ones_col;
  // Streamed FP16 weights: the first a_tmem_k columns of the next layer's A
  // sit in TMEM (from a_col), the rest -- whole 64-column segments, each
  // 128 rows x 128 bytes with the 128-byte swizzle -- in the slot's A buffer
  // in shared memory (sm_a + slot * a_smem_bytes), so that more tile slots
  // fit in TMEM. a_tmem_k covers the widest hidden layer when A fits.
  uint32_t a_tmem_k, sm_a, a_smem_bytes;
  uint32_t stream_w;    // 1: weights streamed through the ring instead of resident
  uint32_t n_wstages;   // streamed-weight ring depth
  uint32_t wstage_bytes;
  // Limits the checking build compares addresses against: the plan's TMEM
  // columns (a test hook may lower it) and the end of its shared-memory
  // layout (bytes from the 1024-aligned base).
  uint32_t chk_tmem_cols, smem_end;
  uint64_t wait_ns;     // limit of every pipeline wait
  uint32_t test_stall;  // non-zero: the MMA thread first waits on kBarNever
};

// Chooses slots, stages and buffers for the network (dims[0..L]) and fills
// the smem plan of `p`. Returns the dynamic smem bytes, or 0 if no plan fits.
uint32_t plan_fused_smem(FusedParams& p, const int32_t* dims, int variant, uint32_t smem_optin);

// `overlap`: launch with programmatic stream serialisation, so that the
// kernel's prologue may overlap the end of the previous kernel on `stream`.
// Only allowed when that previous kernel does not write the packed weights.
cudaError_t launch_fused(const FusedParams& p, int variant, int grid, uint32_t smem,
                         cudaStream_t stream, bool overlap);

// Per-layer offsets of the E4M3 images and the first 16-byte chunk of each
// layer (layers 1..L-1) for the E4M3 packing kernel.
struct Fp8Offsets {
  uint32_t off[kMaxLayers];
  uint32_t chunk_start[kMaxLayers + 1];
};

// E4M3 weight images of the narrow-precision variant (layers 1..L-1, 0-based):
// byte layout of a K-wide FP16 image with K/2 columns, 1024-aligned image
// starts. Requires L >= 2 and hidden widths that are multiples of 32.
// Fills off[l] (l >= 1, relative to the region's start) and returns the
// region's size, or 0 when the network has no such images.
uint32_t fp8_layout(const int32_t* dims, int L, uint32_t* off);

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

// Writes the E4M3 images (fp8_layout) of W_1..W_{L-1} from the packed FP16
// blob p.blob into `region`: each thread rounds 16 weights of one row (round
// to nearest even, saturating at 448) and stores them as one swizzled
// 16-byte chunk.
cudaError_t launch_pack_fp8(const PackParams& p, const uint32_t* fp8_off, uint8_t* region,
                            int num_sms, cudaStream_t stream);

// ---------------------------------------------------------------- host helpers
// Shared by every entry point that launches the kernels (nm_api.cu for the
// handle-based calls, nm_noalloc.cu for the allocation-free one), so that the
// network layout, the tensor maps and the pack parameters have one
// definition.

constexpr int64_t kMaxRows = (static_cast<int64_t>(1) << 31) - 128;  // largest n per dispatch

inline bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// Widths d_0..d_L: 1 <= L <= 16, each a multiple of 16 in [16, 256].
nm_status check_dims(const int32_t* dims, int32_t n_dims);

// Byte offset of each layer's packed image (1024-aligned), element offsets
// of the row-major mirror, and the FP16 biases after the images. Sets p.L and
// p.bias_off; returns the blob's size in bytes. rm_off, rm_b_off and
// mirror_elems may be null.
size_t net_layout(const int32_t* dims, int L, FusedParams& p, uint32_t* w_off, uint32_t* rm_off,
                  uint32_t* rm_b_off, size_t* mirror_elems);

// Kernel parameters that follow from the schedule: the first row of each
// layer's bias among the concatenated biases, each layer's bias-slab offset,
// and their total count.
void set_bias_params(const Schedule& sc, const int32_t* dims, int L, FusedParams& p);

// Input maps [n][d_0] (128-row boxes, one per K-segment width) and output
// maps [n][d_L] (32-row boxes of 32 and/or 16 columns) into p.tm_in / p.tm_out.
nm_status encode_io_maps(FusedParams& p, const int32_t* dims, int L, const void* in, void* out,
                         int64_t n);

// Pack-kernel parameters for a network laid out by net_layout; the row-major
// source (or unpack destination) pointers are left null for the caller.
PackParams make_pack_params(const int32_t* dims, int L, const uint32_t* w_off, uint32_t bias_off,
                            uint8_t* blob);

}  // namespace nm
