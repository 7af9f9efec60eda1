// nm_fused.cu -- persistent fused inference kernel of the FP16 MLP on sm_103a.
//
// One CTA per SM walks 128-sample tiles t = blockIdx.x, blockIdx.x + grid, ...
// and runs every layer of the network on each tile without leaving the SM
// ("Optimization Techniques: Squeezing the Silicon", "Kernel Fusion": one
// write to memory, intermediates stay on chip). Up to five tiles are in
// flight per CTA with resident weights, three with streamed ones (tile
// slots; TMEM decides how many). A slot owns a TMEM region holding its FP32
// accumulator and, beside it, the activations that feed the next layer as
// the tensor core's A operand (FP16 pairs; E4M3 quads in the narrow-precision
// variant; a streamed plan may keep the upper 64-column segments of A in
// shared memory instead, to fit one more slot). The input tile (layer 1's A),
// the weights, the bias operands and the output staging live in shared
// memory. Roles, by warp:
//   epilogue warps  4 x G per slot (the 4 TMEM lane quadrants x G column
//                groups). Per layer they wait for the accumulator, read it
//                (tcgen05.ld), round to FP16, apply max(h, h*half(0.01)) and
//                write the result as the next layer's A -- or, after the last
//                layer, into an output staging tile each warp sends out by
//                TMA -- then meet at the slot's named barrier.
//   issuing lane  one elect.sync lane issues each layer's tcgen05.mma chain,
//                D[128 x N] (FP32, TMEM) = A[128 x K] * W^T + b, and commits
//                it to the slot's accumulator barrier: with resident weights
//                a dedicated warp per slot (it prepares the next chain's
//                descriptors while the epilogue runs); with streamed weights
//                a lane of one of the slot's epilogue warps, which also takes
//                each K-segment from the weight ring.
//   weight producer (streamed weights only): copies the layers' K-segments
//                into the shared weight ring.
//   input producer: keeps every slot's input ring filled by TMA.
//
// The page "Profiling neural material inference" fixes the arithmetic
// ("Experiment setup": the full layer chain per evaluation; "Bad versus good
// activation": the FP16 max form) and supplies the two ablations compiled
// here as variants: "Row-major versus InferencingOptimal weights" (B operand
// rebuilt from row-major memory per tile) and the indexed-lane activation.
//
// With resident weights all UMMA descriptors are precomputed on the host (the
// schedule, one table row per layer) and copied into shared memory once per
// CTA; a layer's chain loads its descriptors together and issues its MMAs as
// straight-line sequences. With streamed weights each 64-wide K-segment's
// descriptors follow from the ring stage it sits in, and its four MMAs are
// issued straight-line too.
//
// Dispatches overlap on a stream: once a CTA holds its tensor memory it lets
// the next kernel be scheduled (programmatic dependent launch), and every
// thread waits on the grid dependency before touching inputs, outputs or the
// status word, so only the prologue runs alongside the previous kernel.
//
// Every wait is bounded by a wall-clock limit. A wait that gives up sets the
// device status word and a CTA-wide abort flag; every role then stops, waits
// (with a fixed limit) for its own copies and MMAs in flight, and the CTA
// frees its tensor memory and exits.
#include <cuda_fp16.h>
#include <cuda_fp8.h>

#include <atomic>
#include <cstring>
#include <mutex>

#include "nm_internal.h"
#include "nm_ptx.cuh"

namespace nm {

namespace {

constexpr uint64_t kDrainNs = 1000000000ull;  // 1 s limit for draining in-flight work

struct Ctx {
  uint32_t sbase;                 // 1024-aligned smem base (shared window address)
  uint32_t bars;                  // shared address of the barrier block
  uint8_t* gbase;                 // generic pointer to the byte at sbase
  volatile uint32_t* abort_flag;  // CTA-wide give-up flag
  uint32_t tmem;                  // TMEM base address
  int32_t n_local;                // tiles this CTA processes
  __device__ __forceinline__ uint32_t bar(int i) const {
    return bars + static_cast<uint32_t>(i) * 8u;
  }
  // Shared-window address of field `off` of layer l's LayerInfo.
  __device__ __forceinline__ uint32_t layer_addr(const FusedParams& p, int l) const {
    return sbase + p.sm_sched + static_cast<uint32_t>(l) * static_cast<uint32_t>(sizeof(LayerInfo));
  }
  __device__ __forceinline__ uint32_t slab_addr(const FusedParams& p, uint32_t j) const {
    return sbase + p.sm_sched + static_cast<uint32_t>(sizeof(LayerInfo) * kMaxLayers) +
           j * static_cast<uint32_t>(sizeof(SlabDesc));
  }
};

__host__ __device__ constexpr bool is_scalar_act(int V) {
  return V == kVarScalar || V == kVarScalarStream;
}

__host__ __device__ constexpr bool is_stream(int V) {
  return V == kVarFusedStream || V == kVarScalarStream || V == kVarFp8Stream ||
         V == kVarFusedStreamSplitA;
}

// Part of the next layer's A may sit in shared memory (a_tmem_k, sm_a).
__host__ __device__ constexpr bool has_split_a(int V) { return V == kVarFusedStreamSplitA; }

// Layers 2..L take E4M3 operands (A: the previous layer's activations,
// rounded as the epilogue stores them; B: the weights' E4M3 images).
__host__ __device__ constexpr bool is_fp8(int V) { return V == kVarFp8Stream; }

// LayerInfo as loaded from shared memory (two 16-byte loads).
struct LayerRegs {
  int32_t K, N;
  uint32_t slab_begin, slab_end, idesc, bslab_off, rm_off, w_off;
};

__device__ __forceinline__ LayerRegs load_layer(const FusedParams& p, const Ctx& c, int l) {
  const uint32_t a = c.layer_addr(p, l);
  const uint4 x = ld_shared_const_u32x4(a), y = ld_shared_const_u32x4(a + 16);
  LayerRegs r;
  r.K = static_cast<int32_t>(x.x);
  r.N = static_cast<int32_t>(x.y);
  r.slab_begin = x.z;
  r.slab_end = x.w;
  r.idesc = y.x;
  r.bslab_off = y.y;
  r.rm_off = y.z;
  r.w_off = y.w;
  return r;
}

// Output width of layer l, from the kernel parameters.
__device__ __forceinline__ int layer_n(const FusedParams& p, int l) {
  return (static_cast<int>((p.n16_bits >> (4 * l)) & 15u) + 1) * 16;
}

__device__ __forceinline__ bool elect_one() {
  uint32_t pred = 0;
  asm volatile("{\n\t.reg .pred P;\n\telect.sync _|P, 0xffffffff;\n\tselp.b32 %0, 1, 0, P;\n\t}" : "=r"(pred));
  return pred != 0;
}

// The checking build (NM_RANGE_CHECKS): every tensor-memory column range a
// warp loads, stores or accumulates into, and every shared-memory range a
// copy or store writes, is compared with the plan's limits before the access;
// a range outside them sets kStatusRangeCheck in the status word (the access
// itself is unchanged). In the normal build these compile to nothing.
//
// Tensor memory: the columns [addr, addr + cols) (relative to the block's
// allocation; the lane bits of addr are ignored) must lie in [lo, hi) and
// below the plan's column count.
__device__ __forceinline__ void chk_tmem(const FusedParams& p, const Ctx& c, uint32_t addr,
                                         uint32_t cols, uint32_t lo, uint32_t hi) {
#ifdef NM_RANGE_CHECKS
  const uint32_t col = (addr & 0xFFFFu) - (c.tmem & 0xFFFFu);
  if (col < lo || col + cols > hi || col + cols > p.chk_tmem_cols)
    atomicOr(p.status, kStatusRangeCheck);
#else
  (void)p, (void)c, (void)addr, (void)cols, (void)lo, (void)hi;
#endif
}

// Tile slot s's accumulator columns, its A columns, and the ones column.
__device__ __forceinline__ void chk_acc(const FusedParams& p, const Ctx& c, uint32_t s,
                                        uint32_t addr, uint32_t cols) {
  chk_tmem(p, c, addr, cols, s * p.slot_cols, s * p.slot_cols + p.a_col);
}
__device__ __forceinline__ void chk_a(const FusedParams& p, const Ctx& c, uint32_t s,
                                      uint32_t addr, uint32_t cols) {
  chk_tmem(p, c, addr, cols, s * p.slot_cols + p.a_col, (s + 1u) * p.slot_cols);
}
__device__ __forceinline__ void chk_ones(const FusedParams& p, const Ctx& c) {
  chk_tmem(p, c, c.tmem + p.ones_col, 8u, p.ones_col, p.ones_col + 32u);
}

__device__ __forceinline__ void chk_smem(const FusedParams& p, const Ctx& c, uint32_t addr,
                                         uint32_t bytes) {
#ifdef NM_RANGE_CHECKS
  if (addr < c.sbase || addr + bytes > c.sbase + p.smem_end) atomicOr(p.status, kStatusRangeCheck);
#else
  (void)p, (void)c, (void)addr, (void)bytes;
#endif
}

// A copy of `bytes` into a buffer of `room` bytes.
__device__ __forceinline__ void chk_fits(const FusedParams& p, uint32_t bytes, uint32_t room) {
#ifdef NM_RANGE_CHECKS
  if (bytes > room) atomicOr(p.status, kStatusRangeCheck);
#else
  (void)p, (void)bytes, (void)room;
#endif
}

// Accumulator columns of an instruction descriptor (its N field).
__device__ __forceinline__ uint32_t idesc_n(uint32_t idesc) { return ((idesc >> 17) & 0x3Fu) << 3; }

// Bounded wait on an mbarrier phase. Gives up (and raises the abort flag and
// the status word) when `limit_ns` passes or another role has given up. The
// abort flag and the clock are looked at once every 64 polls (the clock
// starts at the 64th), so a poll that does not see the phase complete costs
// one try_wait: the flag is in shared memory, and a shared-memory load by a
// warp that has just issued MMAs waits for their operand reads.
__device__ __noinline__ bool wait_phase_slow(uint32_t bar, uint32_t parity, uint64_t limit_ns,
                                             volatile uint32_t* abort_flag, uint32_t* status) {
  uint64_t t0 = 0;
  uint32_t spins = 0;
  while (true) {
    if (mbar_try_wait(bar, parity)) return true;
    if ((++spins & 63u) == 0u) {
      if (*abort_flag) return false;
      const uint64_t now = globaltimer_ns();
      if (spins == 64u) {
        t0 = now;
      } else if (now - t0 > limit_ns) {
        *abort_flag = 1u;
        atomicOr(status, kStatusTimeout);
        return false;
      }
    }
  }
}

__device__ __forceinline__ bool wait_phase(uint32_t bar, uint32_t parity, uint64_t limit_ns,
                                           volatile uint32_t* abort_flag, uint32_t* status) {
  if (mbar_try_wait(bar, parity)) return true;  // fast path, inline
  return wait_phase_slow(bar, parity, limit_ns, abort_flag, status);
}

// Wait used while draining: ignores the abort flag, fixed limit.
__device__ __noinline__ void wait_drain(uint32_t bar, uint32_t parity, uint32_t* status) {
  const uint64_t t0 = globaltimer_ns();
  while (!mbar_try_wait(bar, parity)) {
    if (globaltimer_ns() - t0 > kDrainNs) {
      atomicOr(status, kStatusTimeout);
      return;
    }
  }
}

// Warp-uniform bounded wait: every lane polls, the warp proceeds together.
__device__ __forceinline__ bool warp_wait(uint32_t bar, uint32_t parity, const FusedParams& p,
                                         const Ctx& c) {
  const bool got = wait_phase(bar, parity, p.wait_ns, c.abort_flag, p.status);
  return __all_sync(0xFFFFFFFFu, got);
}

// FP32 accumulator pairs (bias already added by the tensor core) -> FP16
// pairs (round to nearest even), then, for hidden layers (ACT), the
// activation. Column 2j goes to the low half. NP pairs, unrolled.
template <int V, int NP, bool ACT>
__device__ __forceinline__ void convert_pairs(const uint32_t* acc, __half2 slope2, uint32_t* out) {
#pragma unroll
  for (int j = 0; j < NP; ++j) {
    __half2 h = __floats2half2_rn(__uint_as_float(acc[2 * j]), __uint_as_float(acc[2 * j + 1]));
    if (ACT && !is_scalar_act(V)) h = __hmax2(h, __hmul2(h, slope2));
    out[j] = *reinterpret_cast<uint32_t*>(&h);
  }
  if (ACT && is_scalar_act(V)) {
    // The page's indexed-lane form: every FP16 value visited one by one with
    // a dynamic index and a branch.
    __half lanes[2 * NP];
#pragma unroll
    for (int j = 0; j < NP; ++j) {
      __half2 h = *reinterpret_cast<__half2*>(&out[j]);
      lanes[2 * j] = __low2half(h);
      lanes[2 * j + 1] = __high2half(h);
    }
    const __half slope = __low2half(slope2);
    const __half zero = __float2half_rn(0.0f);
#pragma unroll 1
    for (int e = 0; e < 2 * NP; ++e) {
      if (__hlt(lanes[e], zero)) lanes[e] = __hmul(lanes[e], slope);
    }
#pragma unroll
    for (int j = 0; j < NP; ++j) {
      __half2 h = __halves2half2(lanes[2 * j], lanes[2 * j + 1]);
      out[j] = *reinterpret_cast<uint32_t*>(&h);
    }
  }
}

// The narrow-precision variant's hidden-layer epilogue: FP32 accumulator
// pairs -> FP16 pairs (nearest even) -> activation (as convert_pairs) ->
// E4M3 pairs (nearest even, saturating at 448), packed four to a 32-bit
// TMEM column with the lowest K in the lowest byte. NP pairs, NP / 2 words.
template <int NP>
__device__ __forceinline__ void convert_pairs_e4m3(const uint32_t* acc, __half2 slope2,
                                                   uint32_t* out) {
#pragma unroll
  for (int j = 0; j < NP / 2; ++j) {
    __half2 h0 = __floats2half2_rn(__uint_as_float(acc[4 * j]), __uint_as_float(acc[4 * j + 1]));
    __half2 h1 = __floats2half2_rn(__uint_as_float(acc[4 * j + 2]), __uint_as_float(acc[4 * j + 3]));
    h0 = __hmax2(h0, __hmul2(h0, slope2));
    h1 = __hmax2(h1, __hmul2(h1, slope2));
    const uint32_t lo = __nv_cvt_halfraw2_to_fp8x2(static_cast<__half2_raw>(h0), __NV_SATFINITE, __NV_E4M3);
    const uint32_t hi = __nv_cvt_halfraw2_to_fp8x2(static_cast<__half2_raw>(h1), __NV_SATFINITE, __NV_E4M3);
    out[j] = lo | (hi << 16);
  }
}

// A-in-TMEM MMA of one K slab: FP16 operands, or E4M3 ones (F8).
template <bool F8>
__device__ __forceinline__ void umma_ts(uint32_t d, uint32_t a, uint64_t b, uint32_t idesc,
                                        uint32_t accumulate) {
  if constexpr (F8)
    umma_f8_ts(d, a, b, idesc, accumulate);
  else
    umma_f16_ts(d, a, b, idesc, accumulate);
}

// A layer's k-slab MMAs are issued in groups of up to four, each group a
// straight-line sequence with its descriptors already in registers: a
// branch or a dependent load between two MMAs costs the issuing thread far
// more than the MMA itself, and the chain is the slot's critical path. The
// groups keep the code small -- one four-way choice per group instead of a
// fully unrolled sequence per slab count -- which matters because warps that
// sleep at a barrier while others run must find their code still cached.
// Descriptor rows k0 .. k0 + 3 of a layer always lie inside its 16-row block
// of the schedule table, so a group may load all four.
struct PreDesc {
  uint2 b0, b1, b2, b3;
};

__device__ __forceinline__ uint64_t desc_of(uint2 v) {
  return static_cast<uint64_t>(v.y) << 32 | v.x;
}

// B descriptors of slabs k0 .. k0 + 3 (A in TMEM needs no A descriptor).
__device__ __forceinline__ PreDesc load_b4(uint32_t tab, uint32_t k0) {
  const uint32_t a = tab + 16u * k0 + 8u;
  PreDesc d;
  d.b0 = ld_shared_u32x2_ordered(a);
  d.b1 = ld_shared_u32x2_ordered(a + 16u);
  d.b2 = ld_shared_u32x2_ordered(a + 32u);
  d.b3 = ld_shared_u32x2_ordered(a + 48u);
  return d;
}

// A in TMEM (resident-weight layout: slab k of the activations starts 8
// columns, 16 FP16 values per row, after slab k - 1). N MMAs, slabs k0 ...
template <int N>
__device__ __forceinline__ void seq_ts(uint32_t d, uint32_t a_tmem, uint32_t k0, const PreDesc& b,
                                       uint64_t b_add, uint32_t idesc) {
  const uint32_t a = a_tmem + 8u * k0;
  umma_f16_ts(d, a, desc_of(b.b0) + b_add, idesc, k0);
  if (N > 1) umma_f16_ts(d, a + 8u, desc_of(b.b1) + b_add, idesc, 1u);
  if (N > 2) umma_f16_ts(d, a + 16u, desc_of(b.b2) + b_add, idesc, 1u);
  if (N > 3) umma_f16_ts(d, a + 24u, desc_of(b.b3) + b_add, idesc, 1u);
}

__device__ __forceinline__ void group_ts(uint32_t n, uint32_t d, uint32_t a_tmem, uint32_t k0,
                                         const PreDesc& b, uint64_t b_add, uint32_t idesc) {
  switch (n) {
    case 1: seq_ts<1>(d, a_tmem, k0, b, b_add, idesc); break;
    case 2: seq_ts<2>(d, a_tmem, k0, b, b_add, idesc); break;
    case 3: seq_ts<3>(d, a_tmem, k0, b, b_add, idesc); break;
    default: seq_ts<4>(d, a_tmem, k0, b, b_add, idesc); break;
  }
}

// The whole chain on A in TMEM; the first group's descriptors arrive in
// `pre` (fetched before the slot's barrier, off the critical path).
__device__ __forceinline__ void mma_chain_ts(uint32_t nslab, uint32_t d, uint32_t a_tmem,
                                             uint32_t tab, const PreDesc& pre, uint64_t b_add,
                                             uint32_t idesc) {
  group_ts(nslab < 4u ? nslab : 4u, d, a_tmem, 0u, pre, b_add, idesc);
  for (uint32_t k0 = 4; k0 < nslab; k0 += 4) {
    const PreDesc b = load_b4(tab, k0);
    group_ts(nslab - k0 < 4u ? nslab - k0 : 4u, d, a_tmem, k0, b, b_add, idesc);
  }
}

// A in shared memory (layer 1: the input tile): A and B descriptors of
// slabs k0 .. k0 + 3.
struct PreDesc2 {
  uint4 s0, s1, s2, s3;
};

__device__ __forceinline__ PreDesc2 load_ab4(uint32_t tab, uint32_t k0) {
  const uint32_t a = tab + 16u * k0;
  PreDesc2 d;
  d.s0 = ld_shared_u32x4_ordered(a);
  d.s1 = ld_shared_u32x4_ordered(a + 16u);
  d.s2 = ld_shared_u32x4_ordered(a + 32u);
  d.s3 = ld_shared_u32x4_ordered(a + 48u);
  return d;
}

template <int N>
__device__ __forceinline__ void seq_ss(uint32_t d, uint32_t k0, const PreDesc2& s, uint64_t a_add,
                                       uint64_t b_add, uint32_t idesc) {
  umma_f16_ss(d, (static_cast<uint64_t>(s.s0.y) << 32 | s.s0.x) + a_add,
              (static_cast<uint64_t>(s.s0.w) << 32 | s.s0.z) + b_add, idesc, k0);
  if (N > 1)
    umma_f16_ss(d, (static_cast<uint64_t>(s.s1.y) << 32 | s.s1.x) + a_add,
                (static_cast<uint64_t>(s.s1.w) << 32 | s.s1.z) + b_add, idesc, 1u);
  if (N > 2)
    umma_f16_ss(d, (static_cast<uint64_t>(s.s2.y) << 32 | s.s2.x) + a_add,
                (static_cast<uint64_t>(s.s2.w) << 32 | s.s2.z) + b_add, idesc, 1u);
  if (N > 3)
    umma_f16_ss(d, (static_cast<uint64_t>(s.s3.y) << 32 | s.s3.x) + a_add,
                (static_cast<uint64_t>(s.s3.w) << 32 | s.s3.z) + b_add, idesc, 1u);
}

__device__ __forceinline__ void group_ss(uint32_t n, uint32_t d, uint32_t k0, const PreDesc2& s,
                                         uint64_t a_add, uint64_t b_add, uint32_t idesc) {
  switch (n) {
    case 1: seq_ss<1>(d, k0, s, a_add, b_add, idesc); break;
    case 2: seq_ss<2>(d, k0, s, a_add, b_add, idesc); break;
    case 3: seq_ss<3>(d, k0, s, a_add, b_add, idesc); break;
    default: seq_ss<4>(d, k0, s, a_add, b_add, idesc); break;
  }
}

// The chain on the input tile: the first group's descriptors are loaded
// before `wait` (the input tile's arrival) runs, since the table is
// constant. Returns false if `wait` gave up.
template <class Wait>
__device__ __forceinline__ bool mma_chain_ss(uint32_t nslab, uint32_t d, uint32_t tab,
                                             uint64_t a_add, uint64_t b_add, uint32_t idesc,
                                             Wait&& wait) {
  const PreDesc2 first = load_ab4(tab, 0u);
  if (!wait()) return false;
  tc_fence_after_sync();
  group_ss(nslab < 4u ? nslab : 4u, d, 0u, first, a_add, b_add, idesc);
  for (uint32_t k0 = 4; k0 < nslab; k0 += 4) {
    const PreDesc2 s = load_ab4(tab, k0);
    group_ss(nslab - k0 < 4u ? nslab - k0 : 4u, d, k0, s, a_add, b_add, idesc);
  }
  return true;
}

__device__ __forceinline__ void issue_input_tma(const FusedParams& p, uint32_t dst, uint32_t bar,
                                                int32_t tile) {
  const int K = p.d0;
  for (int k = 0; k < K;) {
    uint32_t off;
    int w, k0;
    locate(kTileM, K, k, off, w, k0);
    chk_fits(p, off + kTileM * 2u * static_cast<uint32_t>(w), p.in_stage_bytes);
    tma_load_2d(dst + off, &p.tm_in[swizzle_kind(w)], bar, k0, tile * kTileM);
    k = k0 + w;
  }
}

__device__ __forceinline__ int32_t tile_of(int32_t i) {
  return static_cast<int32_t>(blockIdx.x) + i * static_cast<int32_t>(gridDim.x);
}

// ------------------------------------------------------------------ input producer
// Lane 0 of the producer warp loads the input tiles of all slots in the order
// the slots consume them (tile i goes to slot i % S, round i / S), each into
// its slot's ring stage once the layer-1 MMAs of the round that used the
// stage D rounds earlier have completed. Issuing a TMA load holds the issuing
// thread for hundreds of cycles, so no lane that issues MMAs does it.
__device__ __forceinline__ void run_input_producer(const FusedParams& p, const Ctx& c) {
  const int32_t S = static_cast<int32_t>(p.n_slots);
  const uint32_t D = p.n_in_stages;
  const uint32_t tx = static_cast<uint32_t>(kTileM * 2 * p.d0);
  for (int k = 0; k < 3; ++k) prefetch_tensormap(&p.tm_in[k]);
  bool ok = true;
  int32_t i = 0;
  for (; i < c.n_local && ok; ++i) {
    const int32_t s = i % S;
    const uint32_t r = static_cast<uint32_t>(i / S);
    const uint32_t st = static_cast<uint32_t>(s) * D + r % D;
    ok = wait_phase(c.bar(kBarInEmpty + st), ((r / D) & 1u) ^ 1u, p.wait_ns, c.abort_flag,
                    p.status);
    if (!ok) break;
    mbar_arrive_expect_tx(c.bar(kBarInFull + st), tx);
    chk_smem(p, c, c.sbase + p.sm_in + st * p.in_stage_bytes, p.in_stage_bytes);
    issue_input_tma(p, c.sbase + p.sm_in + st * p.in_stage_bytes, c.bar(kBarInFull + st), tile_of(i));
  }
  // Drain: the loads of the last D rounds of every slot (the latest fill of
  // every stage) must land before the CTA may exit.
  for (int32_t j = i - 1; j >= 0 && j >= i - S * static_cast<int32_t>(D); --j) {
    const uint32_t r = static_cast<uint32_t>(j / S);
    const uint32_t st = static_cast<uint32_t>(j % S) * D + r % D;
    wait_drain(c.bar(kBarInFull + st), (r / D) & 1u, p.status);
  }
}

// Output staging of one tile: a region per 32-column chunk of the output
// (128 rows x 64 bytes, 64-byte swizzle; a trailing 16-column chunk gets
// 128 x 32 bytes, 32-byte swizzle), each 1024-aligned. A warp stores the rows
// of its lane quadrant of its own chunks with its own TMA stores, so no warp
// ever waits for another.
__device__ __forceinline__ uint32_t out_chunk_off(int c0) {
  return static_cast<uint32_t>(c0 >> 5) * (kTileM * 64u);
}

// ------------------------------------------------------------------ streamed weights: slots
// Tile slot s is served by its own 4G warps (4 TMEM lane quadrants x G column
// groups). Per layer evaluation (chain) they wait for the accumulator, round
// and activate it into the slot's A region in TMEM (or, after the last layer,
// into the output staging tile), and meet at the slot's named barrier; then
// one lane of theirs (the issuer) issues the next chain's tcgen05.mma
// sequence and commits it to the slot's accumulator barrier. There is no
// hand-off to another warp between a layer's epilogue and the next layer's
// MMAs: a named barrier costs tens of cycles, an mbarrier hand-off between
// warps a hundred or more. The four or five slots' issuers sit in different
// warps, so their MMA issue latencies overlap.
//
// Every warp of a slot passes the same sequence of named barriers whatever
// happens: a failed wait only turns the remaining work off (`ok`), so no warp
// can be left waiting at a barrier that another has stepped past.
//
// In the row-major ablation the slot's warps also rebuild the next layer's B
// operand from the row-major weights into the slot's B stage before they
// meet (the chain that read the stage has completed by then).
template <int V>
__device__ __forceinline__ void run_slot(const FusedParams& p, const Ctx& c, int warp,
                                                  int lane) {
  const int32_t S = static_cast<int32_t>(p.n_slots);
  const int G = static_cast<int>(p.n_groups);
  const int nw = 4 * G;  // warps of this slot
  const int quad = warp & 3;  // TMEM lane quadrant this warp may access
  // One column group: warp w of group w / 4 serves slot (w / 4 + quad) % S,
  // so each slot has one warp per quadrant and the slots' issuing warps
  // (the lowest-numbered warp of each slot) sit at the lowest warp indices.
  const int32_t s = (G == 1) ? (warp / 4 + quad) % S : warp / nw;
  const int g = (G == 1) ? 0 : (warp % nw) / 4;
  const int wi = (G == 1) ? quad : warp % nw;  // index among the slot's warps
  int iw = 0x7FFFFFFF;
  if (G == 1) {
    for (int qq = 0; qq < 4; ++qq) {
      const int w = 4 * ((s - qq + 4 * S) % S) + qq;
      iw = w < iw ? w : iw;
    }
  }
  const bool issuer_warp = (G == 1) ? (warp == iw) : ((g == 0) && (quad == (s & 3)));
  const bool issuer = issuer_warp && lane == 0;
  const uint32_t row = static_cast<uint32_t>(quad * 32 + lane);
  const uint32_t lane_bits = static_cast<uint32_t>(quad * 32) << 16;
  const uint32_t slot_tmem = c.tmem + static_cast<uint32_t>(s) * p.slot_cols;
  const uint32_t tbase = slot_tmem + lane_bits;
  const uint32_t a_tmem = tbase + p.a_col;
  const uint32_t bar_id = 1u + static_cast<uint32_t>(s);
  const uint32_t bar_threads = 32u * static_cast<uint32_t>(nw);
  const __half2 slope2 = __float2half2_rn(0.01f);  // half(0.01)
  const int L = p.L;
  const int n_out = p.dL;
  const uint32_t D = p.n_in_stages;
  const int32_t n_rounds = (c.n_local - s + S - 1) / S;  // tiles r*S + s < n_local
  const bool storer = (lane == 0) && (32 * g < n_out);
  const uint32_t b_stage = c.sbase + p.sm_b + static_cast<uint32_t>(s) * p.b_stage_bytes;
  const uint32_t a_smem =
      has_split_a(V) ? c.sbase + p.sm_a + static_cast<uint32_t>(s) * p.a_smem_bytes : 0u;

  // Row-major ablation: this warp's share (rows wi, wi + nw, ...) of W_l
  // rebuilt in the slot's B stage, 16-byte loads, swizzled 16-byte stores.
  auto rebuild_b = [&](int l) {
    const LayerRegs li = load_layer(p, c, l);
    const int K = li.K, N = li.N, kc = K >> 3;
    const uint16_t* Wl = p.mirror + li.rm_off;
    for (int idx = wi * 32 + lane; idx < N * kc; idx += 32 * nw) {
      const int n = idx / kc, col = (idx - n * kc) << 3;
      const uint4 v = __ldg(reinterpret_cast<const uint4*>(Wl + n * K + col));
      uint32_t off;
      int w, k0;
      locate(static_cast<uint32_t>(N), K, col, off, w, k0);
      chk_smem(p, c, b_stage + off + swz(static_cast<uint32_t>(n * 2 * w + (col - k0) * 2), w), 16u);
      st_shared_v4(b_stage + off + swz(static_cast<uint32_t>(n * 2 * w + (col - k0) * 2), w), v.x,
                   v.y, v.z, v.w);
    }
    fence_proxy_async_smem();  // generic-proxy stores -> MMA reads (async proxy)
  };

  // The issuer: chain (round rr, layer l). Layer 1 reads the input tile in
  // shared memory once it has landed; later layers read A from TMEM. The
  // bias MMA (ones slab x bias slab) closes every chain.
  // Streamed weights: the next weight-ring stage to consume and the parity
  // of its current fill (kept by the issuing lane only).
  uint32_t ws = 0, wph = 0;
  auto next_stage = [&]() {
    if (++ws == p.n_wstages) {
      ws = 0;
      wph ^= 1u;
    }
  };
  // Streamed weights: the layer's K-segments are taken from the ring as the
  // weight-producer warp fills it, in the (round, layer, segment) order in
  // which every slot consumes it, one segment per stage; each stage is
  // released by a commit once this slot's MMAs on it complete.
  auto issue_stream = [&](int32_t rr, int l) -> bool {
    const LayerRegs li = load_layer(p, c, l);
    const uint32_t st = static_cast<uint32_t>(s) * D + static_cast<uint32_t>(rr) % D;
    const uint32_t in_base = c.sbase + p.sm_in + st * p.in_stage_bytes;
    chk_acc(p, c, static_cast<uint32_t>(s), slot_tmem, idesc_n(li.idesc));
    chk_ones(p, c);
    if (l == 0) {
      chk_smem(p, c, in_base, p.in_stage_bytes);
    } else {
      const uint32_t k_tm = (has_split_a(V) && static_cast<uint32_t>(li.K) > p.a_tmem_k)
                                ? p.a_tmem_k : static_cast<uint32_t>(li.K);
      chk_a(p, c, static_cast<uint32_t>(s), slot_tmem + p.a_col, k_tm >> 1);
      if (has_split_a(V) && static_cast<uint32_t>(li.K) > p.a_tmem_k)
        chk_smem(p, c, a_smem, 256u * (static_cast<uint32_t>(li.K) - p.a_tmem_k));
    }
    bool ok = true;
    if (l == 0)
      ok = wait_phase(c.bar(kBarInFull + st), (static_cast<uint32_t>(rr) / D) & 1u, p.wait_ns,
                      c.abort_flag, p.status);
    // 64-wide K-segments (all of them when K is a multiple of 64): the four
    // k-slab MMAs of each are issued straight-line, with the segment's
    // descriptors derived from its ring stage alone -- segment j of the
    // input tile starts 128 x 128 bytes after segment j - 1, and the layer's
    // A in TMEM 32 columns after.
    const int n64 = li.K >> 6;
    const uint64_t desc64 = smem_desc(0u, 1024u, swizzle_code(64));
    if (l == 0) {
      for (int j = 0; j < n64 && ok; ++j) {
        ok = wait_phase(c.bar(kBarWFull + ws), wph, p.wait_ns, c.abort_flag, p.status);
        if (!ok) break;
        tc_fence_after_sync();
        const uint64_t bd = desc64 + ((c.sbase + p.sm_wring + ws * p.wstage_bytes) >> 4);
        const uint64_t ad = desc64 + ((in_base + 16384u * static_cast<uint32_t>(j)) >> 4);
        umma_f16_ss(slot_tmem, ad, bd, li.idesc, j > 0 ? 1u : 0u);
        umma_f16_ss(slot_tmem, ad + 2u, bd + 2u, li.idesc, 1u);
        umma_f16_ss(slot_tmem, ad + 4u, bd + 4u, li.idesc, 1u);
        umma_f16_ss(slot_tmem, ad + 6u, bd + 6u, li.idesc, 1u);
        umma_commit(c.bar(kBarWEmpty + ws));
        next_stage();
      }
    } else {
      for (int j = 0; j < n64 && ok; ++j) {
        ok = wait_phase(c.bar(kBarWFull + ws), wph, p.wait_ns, c.abort_flag, p.status);
        if (!ok) break;
        tc_fence_after_sync();
        const uint64_t bd = desc64 + ((c.sbase + p.sm_wring + ws * p.wstage_bytes) >> 4);
        const uint32_t kj = 64u * static_cast<uint32_t>(j);
        if (!has_split_a(V) || kj < p.a_tmem_k) {
          const uint32_t at = slot_tmem + p.a_col + (kj >> 1);
          umma_ts<is_fp8(V)>(slot_tmem, at, bd, li.idesc, j > 0 ? 1u : 0u);
          umma_ts<is_fp8(V)>(slot_tmem, at + 8u, bd + 2u, li.idesc, 1u);
          umma_ts<is_fp8(V)>(slot_tmem, at + 16u, bd + 4u, li.idesc, 1u);
          umma_ts<is_fp8(V)>(slot_tmem, at + 24u, bd + 6u, li.idesc, 1u);
        } else {
          // this segment of A is in the slot's shared-memory A buffer
          const uint64_t ad = desc64 + ((a_smem + 128u * (kj - p.a_tmem_k) * 2u) >> 4);
          umma_f16_ss(slot_tmem, ad, bd, li.idesc, j > 0 ? 1u : 0u);
          umma_f16_ss(slot_tmem, ad + 2u, bd + 2u, li.idesc, 1u);
          umma_f16_ss(slot_tmem, ad + 4u, bd + 4u, li.idesc, 1u);
          umma_f16_ss(slot_tmem, ad + 6u, bd + 6u, li.idesc, 1u);
        }
        umma_commit(c.bar(kBarWEmpty + ws));
        next_stage();
      }
    }
    // The narrower tail segments (K mod 64 = 16, 32 or 48).
    for (int k = n64 << 6; k < li.K && ok;) {
      uint32_t aoff;
      int w, k0;
      locate(kTileM, li.K, k, aoff, w, k0);
      ok = wait_phase(c.bar(kBarWFull + ws), wph, p.wait_ns, c.abort_flag, p.status);
      if (!ok) break;
      tc_fence_after_sync();
      // One K-segment: w / 16 k-slabs, 32 bytes apart in the segment's
      // swizzle atom, so slab j's descriptors are the segment's plus 2j
      // (start addresses are in 16-byte units). Issued straight-line.
      const uint32_t sbo = 16u * static_cast<uint32_t>(w);
      const uint32_t swc = swizzle_code(w);
      const uint64_t bd = smem_desc(c.sbase + p.sm_wring + ws * p.wstage_bytes, sbo, swc);
      const uint32_t acc0 = static_cast<uint32_t>(k0);  // the layer's first slab overwrites
      if (l == 0) {
        const uint64_t ad = smem_desc(in_base + aoff, sbo, swc);
        umma_f16_ss(slot_tmem, ad, bd, li.idesc, acc0);
        if (w >= 32) umma_f16_ss(slot_tmem, ad + 2u, bd + 2u, li.idesc, 1u);
        if (w == 64) {
          umma_f16_ss(slot_tmem, ad + 4u, bd + 4u, li.idesc, 1u);
          umma_f16_ss(slot_tmem, ad + 6u, bd + 6u, li.idesc, 1u);
        }
      } else {
        const uint32_t at = slot_tmem + p.a_col + (static_cast<uint32_t>(k0) >> 1);
        umma_ts<is_fp8(V)>(slot_tmem, at, bd, li.idesc, acc0);
        if (w >= 32) umma_ts<is_fp8(V)>(slot_tmem, at + 8u, bd + 2u, li.idesc, 1u);
        if (w == 64) {
          umma_ts<is_fp8(V)>(slot_tmem, at + 16u, bd + 4u, li.idesc, 1u);
          umma_ts<is_fp8(V)>(slot_tmem, at + 24u, bd + 6u, li.idesc, 1u);
        }
      }
      umma_commit(c.bar(kBarWEmpty + ws));
      next_stage();
      k = k0 + w;
    }
    if (ok) {
      umma_f16_ts(slot_tmem, c.tmem + p.ones_col,
                  smem_desc(c.sbase + p.sm_bslab + li.bslab_off, 256u, 6u), li.idesc, 1u);
      umma_commit(c.bar(kBarAccFull + s));
      if (l == 0) umma_commit(c.bar(kBarInEmpty + st));
    }
    return ok;
  };
  auto issue = [&](int32_t rr, int l) -> bool {
    if constexpr (is_stream(V)) return issue_stream(rr, l);
    const LayerRegs li = load_layer(p, c, l);
    const uint32_t st = static_cast<uint32_t>(s) * D + static_cast<uint32_t>(rr) % D;
    const uint32_t b_base = (V == kVarRowMajor) ? b_stage : c.sbase + p.sm_w + li.w_off;
    const uint64_t b_add = b_base >> 4;
    // Slab count from the kernel parameters and the table row by layer: the
    // descriptor loads do not wait for the layer entry.
    const uint32_t nslab = static_cast<uint32_t>((p.nslab_bits >> (4 * l)) & 15u) + 1u;
    const uint32_t tab = c.slab_addr(p, 16u * static_cast<uint32_t>(l));
    const uint64_t bias_bd = smem_desc(c.sbase + p.sm_bslab + li.bslab_off, 256u, 6u);
    bool ok = true;
    if (l == 0) {
      const uint64_t a_add = (c.sbase + p.sm_in + st * p.in_stage_bytes) >> 4;
      auto wait = [&]() -> bool {
        return wait_phase(c.bar(kBarInFull + st), (static_cast<uint32_t>(rr) / D) & 1u, p.wait_ns,
                          c.abort_flag, p.status);
      };
      ok = mma_chain_ss(nslab, slot_tmem, tab, a_add, b_add, li.idesc, wait);
    } else {
      tc_fence_after_sync();
      mma_chain_ts(nslab, slot_tmem, slot_tmem + p.a_col, tab, load_b4(tab, 0u), b_add, li.idesc);
    }
    if (ok) {
      umma_f16_ts(slot_tmem, c.tmem + p.ones_col, bias_bd, li.idesc, 1u);
      umma_commit(c.bar(kBarAccFull + s));
      if (l == 0) umma_commit(c.bar(kBarInEmpty + st));
    }
    return ok;
  };

  bool ok = warp_wait(c.bar(kBarWLoad), 0, p, c);
  if (issuer_warp) {
    bool iok = ok;
    if (issuer && iok && p.test_stall)
      iok = wait_phase(c.bar(kBarNever), 0, p.wait_ns, c.abort_flag, p.status);
    ok = __shfl_sync(0xFFFFFFFFu, iok, 0);
  }
  if (n_rounds > 0) {
    if (V == kVarRowMajor && ok) rebuild_b(0);
    named_bar_sync(bar_id, bar_threads);
    if (issuer_warp) {
      bool iok = ok;
      if (iok && elect_one()) iok = issue(0, 0);
      ok = __shfl_sync(0xFFFFFFFFu, iok, 0);
    }
  }
  for (int32_t r = 0; r < n_rounds; ++r) {
    const int32_t t = tile_of(r * S + s);
    // Hidden layers: accumulator -> FP16 -> activation -> next layer's A.
    for (int l = 0; l < L - 1; ++l) {
      const uint32_t q = static_cast<uint32_t>(r * L + l);
      // The width comes from the kernel parameters, not from the schedule in
      // shared memory: a shared-memory load issued by the warp that has just
      // issued the previous chain's MMAs waits until those MMAs have read
      // their shared-memory operands, which would hold that warp back.
      const int N = layer_n(p, l);
      bool a_in_smem = false;  // (split-A plans) a chunk went to shared memory
      if (ok) ok = warp_wait(c.bar(kBarAccFull + s), q & 1u, p, c);
      if (ok) {
        tc_fence_after_sync();
        for (int c0 = 32 * g; c0 + 32 <= N; c0 += 32 * G) {
          uint32_t acc[32];
          chk_acc(p, c, static_cast<uint32_t>(s), tbase + static_cast<uint32_t>(c0), 32u);
          tmem_ld_x32(tbase + static_cast<uint32_t>(c0), acc);
          tmem_wait_ld();
          if constexpr (is_fp8(V)) {
            uint32_t q[8];
            convert_pairs_e4m3<16>(acc, slope2, q);
            chk_a(p, c, static_cast<uint32_t>(s), a_tmem + static_cast<uint32_t>(c0 >> 2), 8u);
            tmem_st_x8(a_tmem + static_cast<uint32_t>(c0 >> 2), q);
          } else {
            uint32_t h[16];
            convert_pairs<V, 16, true>(acc, slope2, h);
            if (!has_split_a(V) || static_cast<uint32_t>(c0) < p.a_tmem_k) {
              chk_a(p, c, static_cast<uint32_t>(s), a_tmem + static_cast<uint32_t>(c0 >> 1), 16u);
              tmem_st_x16(a_tmem + static_cast<uint32_t>(c0 >> 1), h);
            } else {
              // this row's 64 bytes of the chunk, into the 128-byte-swizzled
              // 64-column segment of the shared-memory A buffer (a layer
              // wider than a_tmem_k is a multiple of 64 wide)
              const uint32_t kk = static_cast<uint32_t>(c0) - p.a_tmem_k;
              const uint32_t base = a_smem + (kk >> 6) * (kTileM * 128u);
#pragma unroll
              for (int cc = 0; cc < 4; ++cc) {
                chk_smem(p, c, base + swz(row * 128u + (kk & 63u) * 2u + 16u * cc, 64), 16u);
                st_shared_v4(base + swz(row * 128u + (kk & 63u) * 2u + 16u * cc, 64), h[4 * cc],
                             h[4 * cc + 1], h[4 * cc + 2], h[4 * cc + 3]);
              }
              a_in_smem = true;
            }
          }
        }
        // (hidden widths of the narrow-precision variant are multiples of 32)
        if (!is_fp8(V) && (N & 31) && ((N >> 5) % G) == g) {
          const int c0 = N - 16;
          uint32_t acc[16], h[8];
          chk_acc(p, c, static_cast<uint32_t>(s), tbase + static_cast<uint32_t>(c0), 16u);
          tmem_ld_x16(tbase + static_cast<uint32_t>(c0), acc);
          tmem_wait_ld();
          convert_pairs<V, 8, true>(acc, slope2, h);
          chk_a(p, c, static_cast<uint32_t>(s), a_tmem + static_cast<uint32_t>(c0 >> 1), 8u);
          tmem_st_x8(a_tmem + static_cast<uint32_t>(c0 >> 1), h);
        }
        if (V == kVarRowMajor) rebuild_b(l + 1);
        // generic-proxy stores -> the next chain's MMA reads (async proxy)
        if (has_split_a(V) && a_in_smem) fence_proxy_async_smem();
        tmem_wait_st();
      }
      tc_fence_before_sync();
      named_bar_sync(bar_id, bar_threads);
      if (issuer_warp) {
        bool iok = ok;
        if (iok && elect_one()) iok = issue(r, l + 1);
        ok = __shfl_sync(0xFFFFFFFFu, iok, 0);
      }
    }
    // Last layer: accumulator -> FP16 -> output staging -> TMA store; the
    // slot then starts its next tile.
    {
      const int l = L - 1;
      const uint32_t q = static_cast<uint32_t>(r * L + l);
      const int N = n_out;
      const uint32_t out_dst =
          c.sbase + p.sm_out +
          (static_cast<uint32_t>(s) * p.n_out_bufs + static_cast<uint32_t>(r) % p.n_out_bufs) *
              p.out_slot_bytes;
      // This staging buffer went to this warp's TMA stores n_out_bufs tiles
      // of this slot ago; they must have finished reading it (checked before
      // the accumulator wait, which it does not depend on).
      if (storer) {
        if (p.n_out_bufs > 1)
          bulk_wait_group_read<1>();
        else
          bulk_wait_group_read<0>();
      }
      __syncwarp();
      if (ok) ok = warp_wait(c.bar(kBarAccFull + s), q & 1u, p, c);
      if (ok) {
        tc_fence_after_sync();
        for (int c0 = 32 * g; c0 + 32 <= N; c0 += 32 * G) {
          uint32_t acc[32], h[16];
          chk_acc(p, c, static_cast<uint32_t>(s), tbase + static_cast<uint32_t>(c0), 32u);
          tmem_ld_x32(tbase + static_cast<uint32_t>(c0), acc);
          tmem_wait_ld();
          convert_pairs<V, 16, false>(acc, slope2, h);
          const uint32_t base = out_dst + out_chunk_off(c0);
#pragma unroll
          for (int cc = 0; cc < 4; ++cc) {
            chk_smem(p, c, base + swz(row * 64u + cc * 16u, 32), 16u);
            st_shared_v4_nc(base + swz(row * 64u + cc * 16u, 32), h[4 * cc], h[4 * cc + 1],
                            h[4 * cc + 2], h[4 * cc + 3]);
          }
        }
        if ((N & 31) && ((N >> 5) % G) == g) {
          const int c0 = N - 16;
          uint32_t acc[16], h[8];
          chk_acc(p, c, static_cast<uint32_t>(s), tbase + static_cast<uint32_t>(c0), 16u);
          tmem_ld_x16(tbase + static_cast<uint32_t>(c0), acc);
          tmem_wait_ld();
          convert_pairs<V, 8, false>(acc, slope2, h);
          const uint32_t base = out_dst + out_chunk_off(c0);
#pragma unroll
          for (int cc = 0; cc < 2; ++cc) {
            chk_smem(p, c, base + swz(row * 32u + cc * 16u, 16), 16u);
            st_shared_v4_nc(base + swz(row * 32u + cc * 16u, 16), h[4 * cc], h[4 * cc + 1],
                            h[4 * cc + 2], h[4 * cc + 3]);
          }
        }
        if (V == kVarRowMajor && (r + 1) * S + s < c.n_local) rebuild_b(0);
        fence_proxy_async_smem();  // staging tile -> TMA store (async proxy)
      }
      tc_fence_before_sync();
      named_bar_sync(bar_id, bar_threads);
      if (issuer_warp) {
        bool iok = ok;
        if (iok && r + 1 < n_rounds && elect_one()) iok = issue(r + 1, 0);
        ok = __shfl_sync(0xFFFFFFFFu, iok, 0);
      }
      if (storer && ok) {
        const int64_t row0 = static_cast<int64_t>(t) * kTileM + quad * 32;
        if (row0 < p.n) {
          for (int c0 = 32 * g; c0 < N; c0 += 32 * G) {
            const int cols = (N - c0 >= 32) ? 32 : 16;
            tma_store_2d(&p.tm_out[swizzle_kind(cols)],
                         out_dst + out_chunk_off(c0) + static_cast<uint32_t>(quad * 32 * 2 * cols),
                         c0, static_cast<int32_t>(row0));
          }
        }
      }
      if (storer) bulk_commit_group();
    }
  }
  if constexpr (is_stream(V)) {
    // Rounds in which this slot has no tile: its share of releasing every
    // weight-ring stage, without MMAs.
    if (issuer_warp && ok && elect_one()) {
      const int32_t n_rounds_all = (c.n_local + S - 1) / S;
      bool wok = true;
      for (int32_t r = n_rounds; r < n_rounds_all && wok; ++r) {
        for (int l = 0; l < L && wok; ++l) {
          const LayerRegs li = load_layer(p, c, l);
          for (int k = 0; k < li.K && wok;) {
            uint32_t off;
            int w, k0;
            locate(kTileM, li.K, k, off, w, k0);
            wok = wait_phase(c.bar(kBarWFull + ws), wph, p.wait_ns, c.abort_flag, p.status);
            if (wok) mbar_arrive(c.bar(kBarWEmpty + ws));
            next_stage();
            k = k0 + w;
          }
        }
      }
    }
    __syncwarp();
  }
  if (issuer) {
    // Drain: every MMA this thread issued completes before the CTA may exit.
    umma_commit(c.bar(kBarDrain + s));
    wait_drain(c.bar(kBarDrain + s), 0, p.status);
  }
  if (storer) bulk_wait_group_all();
}

// ------------------------------------------------------------------ resident weights
// With resident weights each tile slot has one issuing warp and 4G epilogue
// warps that meet at the slot's named barrier once per layer evaluation
// (chain): the epilogue warps arrive when they have turned the accumulator
// into the next layer's A (or into the output staging tile), the issuing
// warp arrives when it is ready to issue the next chain. A warp that issues
// MMAs stays busy for several hundred cycles after its commit (the MMAs'
// issue, the warp's reconvergence, the loop), so the issuing warp does no
// epilogue work: its overhead runs while the epilogue warps work, and all of
// them wait for the accumulator together instead of one of them arriving
// late at every layer.
//
// Both sides pass the same sequence of barriers whatever happens (one at the
// start, one after every chain's epilogue): a failed wait only turns the
// remaining work off (`ok`), so no warp is ever left at a barrier that the
// others have stepped past. A wait that gives up raises the CTA's abort
// flag, which ends the other side's waits too.

// The issuing warp of slot s: issues chain (r, l) -- K/16 MMAs plus the bias
// MMA, committed to the slot's accumulator barrier -- after the barrier that
// follows chain (r, l - 1)'s epilogue (or, for l = 0, round r - 1's last
// epilogue). Layer 1 reads the input tile from shared memory once it has
// landed; later layers read A from TMEM, and their descriptors are fetched
// before the barrier.
template <int V>
__device__ __forceinline__ void run_issuer(const FusedParams& p, const Ctx& c, int32_t g, int lane) {
  const int32_t S = static_cast<int32_t>(p.n_slots);
  const int L = p.L;
  const uint32_t D = p.n_in_stages;
  const int32_t s0 = static_cast<int32_t>(p.grp_first[g]);  // the group's first tile region
  const int32_t T = static_cast<int32_t>(p.grp_tiles[g]);   // its regions (1 or 2)
  const int32_t n_rounds = (c.n_local - s0 + S - 1) / S;    // rounds with a tile in region s0
  const uint32_t bar_id = 1u + static_cast<uint32_t>(g);
  const uint32_t bar_threads = 32u * (4u * p.n_groups * static_cast<uint32_t>(T) + 1u);
  auto tmem_of = [&](int32_t s) { return c.tmem + static_cast<uint32_t>(s) * p.slot_cols; };
  auto b_stage_of = [&](int32_t s) {
    return c.sbase + p.sm_b + static_cast<uint32_t>(s) * p.b_stage_bytes;
  };

  // Everything a chain on A in TMEM needs that does not depend on the
  // epilogue -- the layer's entry and its first B descriptors -- shared by
  // the group's regions (same layer, same weights). The first group's B
  // descriptors are complete (base added), so that after the barrier only
  // the MMAs and the commits remain.
  struct IssuePrep {
    uint64_t b_add, bias_bd;
    uint32_t idesc, nslab, tab;
    PreDesc bd;
  };
  auto prep_ts = [&](int l) -> IssuePrep {
    IssuePrep ip;
    const LayerRegs li = load_layer(p, c, l);
    ip.idesc = li.idesc;
    ip.b_add = ((V == kVarRowMajor) ? b_stage_of(s0) : c.sbase + p.sm_w + li.w_off) >> 4;
    ip.bias_bd = smem_desc(c.sbase + p.sm_bslab + li.bslab_off, 256u, 6u);
    ip.nslab = static_cast<uint32_t>((p.nslab_bits >> (4 * l)) & 15u) + 1u;
    ip.tab = c.slab_addr(p, 16u * static_cast<uint32_t>(l));
    ip.bd = load_b4(ip.tab, 0u);
    auto add = [&](uint2& v) {
      const uint64_t d = desc_of(v) + ip.b_add;
      v.x = static_cast<uint32_t>(d);
      v.y = static_cast<uint32_t>(d >> 32);
    };
    add(ip.bd.b0);
    add(ip.bd.b1);
    add(ip.bd.b2);
    add(ip.bd.b3);
    return ip;
  };
  // Chain of region s (A in TMEM). In the row-major ablation each region
  // has its own B stage, so the second region's descriptors are rebased.
  auto fire_ts = [&](const IssuePrep& ip, int32_t s) {
    const uint32_t d = tmem_of(s);
    const uint32_t a = d + p.a_col;
    uint64_t b_add = ip.b_add;
    PreDesc bd = ip.bd;
    if (V == kVarRowMajor && s != s0) {
      const uint64_t delta = static_cast<uint64_t>((b_stage_of(s) - b_stage_of(s0)) >> 4);
      b_add += delta;
      auto add = [&](uint2& v) {
        const uint64_t x = desc_of(v) + delta;
        v.x = static_cast<uint32_t>(x);
        v.y = static_cast<uint32_t>(x >> 32);
      };
      add(bd.b0);
      add(bd.b1);
      add(bd.b2);
      add(bd.b3);
    }
    chk_acc(p, c, static_cast<uint32_t>(s), d, idesc_n(ip.idesc));
    chk_a(p, c, static_cast<uint32_t>(s), a, 8u * ip.nslab);
    chk_ones(p, c);
    group_ts(ip.nslab < 4u ? ip.nslab : 4u, d, a, 0u, bd, 0u, ip.idesc);
    for (uint32_t k0 = 4; k0 < ip.nslab; k0 += 4) {
      const PreDesc b = load_b4(ip.tab, k0);
      group_ts(ip.nslab - k0 < 4u ? ip.nslab - k0 : 4u, d, a, k0, b, b_add, ip.idesc);
    }
    umma_f16_ts(d, c.tmem + p.ones_col, ip.bias_bd, ip.idesc, 1u);
    umma_commit(c.bar(kBarAccFull + s));
  };
  // Layer 1 of round rr in region s: A is the input tile in the region's
  // ring stage.
  auto issue_first = [&](int32_t rr, int32_t s) -> bool {
    const LayerRegs li = load_layer(p, c, 0);
    const uint32_t st = static_cast<uint32_t>(s) * D + static_cast<uint32_t>(rr) % D;
    const uint32_t b_base = (V == kVarRowMajor) ? b_stage_of(s) : c.sbase + p.sm_w + li.w_off;
    const uint32_t nslab = static_cast<uint32_t>(p.nslab_bits & 15u) + 1u;
    const uint64_t a_add = (c.sbase + p.sm_in + st * p.in_stage_bytes) >> 4;
    auto wait = [&]() -> bool {
      return wait_phase(c.bar(kBarInFull + st), (static_cast<uint32_t>(rr) / D) & 1u, p.wait_ns,
                        c.abort_flag, p.status);
    };
    const uint32_t d = tmem_of(s);
    chk_acc(p, c, static_cast<uint32_t>(s), d, idesc_n(li.idesc));
    chk_smem(p, c, c.sbase + p.sm_in + st * p.in_stage_bytes, p.in_stage_bytes);
    if (!mma_chain_ss(nslab, d, c.slab_addr(p, 0u), a_add, b_base >> 4, li.idesc, wait))
      return false;
    umma_f16_ts(d, c.tmem + p.ones_col, smem_desc(c.sbase + p.sm_bslab + li.bslab_off, 256u, 6u),
                li.idesc, 1u);
    umma_commit(c.bar(kBarAccFull + s));
    umma_commit(c.bar(kBarInEmpty + st));
    return true;
  };

  bool ok = warp_wait(c.bar(kBarWLoad), 0, p, c);
  if (ok && p.test_stall) {
    bool iok = true;
    if (lane == 0) iok = wait_phase(c.bar(kBarNever), 0, p.wait_ns, c.abort_flag, p.status);
    ok = __shfl_sync(0xFFFFFFFFu, iok, 0);
  }
  if (n_rounds > 0) {
    named_bar_sync(bar_id, bar_threads);  // the epilogue warps are set up
    IssuePrep ip;
    for (int32_t r = 0; r < n_rounds; ++r) {
      // the group's regions that hold a tile this round (the last round may
      // be partial)
      const int32_t nt = (r * S + s0 + T <= c.n_local) ? T : c.n_local - (r * S + s0);
      for (int l = 0; l < L; ++l) {
        // Chain (r, l) of each of the group's tiles ...
        if (l == 0) {
          if (ok) {
            bool iok = true;
            if (elect_one()) {
              for (int32_t t = 0; t < nt && iok; ++t) iok = issue_first(r, s0 + t);
            }
            ok = __all_sync(0xFFFFFFFFu, iok);
          }
        } else if (ok && elect_one()) {
          fire_ts(ip, s0);
          if (nt > 1) fire_ts(ip, s0 + 1);
        }
        // ... then, while their epilogue runs, the next chain's descriptors
        // (layers after the first), and the barrier after that epilogue. The
        // warp is not reconverged after the elected lane's issue: its other
        // lanes go ahead, so the barrier is the per-thread form.
        if (l + 1 < L) ip = prep_ts(l + 1);
        tc_fence_before_sync();
        named_bar_sync_lanes(bar_id, bar_threads);
        // the epilogue's tcgen05.st of the next A (waited and fenced before
        // the barrier) -> this warp's next MMAs, which read it
        tc_fence_after_sync();
      }
    }
  }
  // Drain: every MMA this warp issued completes before the CTA may exit (the
  // lane elect.sync picks here is the one that issued them).
  if (elect_one()) {
    umma_commit(c.bar(kBarDrain + g));
    wait_drain(c.bar(kBarDrain + g), 0, p.status);
  }
  __syncwarp();
}

// Epilogue warp e of the resident-weight roles (slot e / 4G, lane quadrant
// e % 4, column group (e % 4G) / 4): per chain it waits for the slot's
// accumulator, reads its columns (tcgen05.ld), rounds to FP16 and applies
// max(h, h * half(0.01)) for a hidden layer, writing the FP16 pairs as the
// next layer's A (tcgen05.st); after the last layer it writes its rows into
// the output staging tile and sends them out by TMA once the slot has met.
template <int V>
__device__ __forceinline__ void run_epilogue(const FusedParams& p, const Ctx& c, int e, int lane) {
  const int32_t S = static_cast<int32_t>(p.n_slots);
  const int G = static_cast<int>(p.n_groups);
  const int nw = 4 * G;             // epilogue warps of a slot
  const int32_t s = e / nw;
  const int wi = e % nw;            // index among the slot's epilogue warps
  const int g = wi / 4;             // column group
  const int quad = e & 3;           // TMEM lane quadrant (kEpiWarp0 is a multiple of 4)
  const uint32_t row = static_cast<uint32_t>(quad * 32 + lane);
  const uint32_t lane_bits = static_cast<uint32_t>(quad * 32) << 16;
  const uint32_t tbase = c.tmem + static_cast<uint32_t>(s) * p.slot_cols + lane_bits;
  const uint32_t a_tmem = tbase + p.a_col;
  const uint32_t grp = p.grp_of[s];
  const int32_t s0 = static_cast<int32_t>(p.grp_first[grp]);
  const uint32_t bar_id = 1u + grp;
  const uint32_t bar_threads = 32u * static_cast<uint32_t>(nw) * p.grp_tiles[grp] + 32u;
  const __half2 slope2 = __float2half2_rn(0.01f);  // half(0.01)
  const int L = p.L;
  const int n_out = p.dL;
  // The group's rounds (those of its first region); this region holds a tile
  // in all of them but possibly the last.
  const int32_t n_rounds = (c.n_local - s0 + S - 1) / S;
  const bool storer = (lane == 0) && (32 * g < n_out);
  const uint32_t b_stage = c.sbase + p.sm_b + static_cast<uint32_t>(s) * p.b_stage_bytes;

  // Row-major ablation: this warp's share (rows wi, wi + nw, ...) of W_l
  // rebuilt in the slot's B stage, 16-byte loads, swizzled 16-byte stores.
  auto rebuild_b = [&](int l) {
    const LayerRegs li = load_layer(p, c, l);
    const int K = li.K, N = li.N, kc = K >> 3;
    const uint16_t* Wl = p.mirror + li.rm_off;
    for (int idx = wi * 32 + lane; idx < N * kc; idx += 32 * nw) {
      const int n = idx / kc, col = (idx - n * kc) << 3;
      const uint4 v = __ldg(reinterpret_cast<const uint4*>(Wl + n * K + col));
      uint32_t off;
      int w, k0;
      locate(static_cast<uint32_t>(N), K, col, off, w, k0);
      chk_smem(p, c, b_stage + off + swz(static_cast<uint32_t>(n * 2 * w + (col - k0) * 2), w), 16u);
      st_shared_v4(b_stage + off + swz(static_cast<uint32_t>(n * 2 * w + (col - k0) * 2), w), v.x,
                   v.y, v.z, v.w);
    }
    fence_proxy_async_smem();  // generic-proxy stores -> MMA reads (async proxy)
  };

  bool ok = warp_wait(c.bar(kBarWLoad), 0, p, c);
  if (n_rounds > 0) {
    if (V == kVarRowMajor && ok) rebuild_b(0);
    named_bar_sync(bar_id, bar_threads);
  }
  for (int32_t r = 0; r < n_rounds; ++r) {
    const int32_t t = tile_of(r * S + s);
    const bool has = r * S + s < c.n_local;  // else: pass the group's barriers only
    // Hidden layers: accumulator -> FP16 -> activation -> next layer's A.
    for (int l = 0; l < L - 1; ++l) {
      const uint32_t q = static_cast<uint32_t>(r * L + l);
      const int N = layer_n(p, l);
      if (ok && has) ok = warp_wait(c.bar(kBarAccFull + s), q & 1u, p, c);
      if (ok && has) {
        tc_fence_after_sync();
        for (int c0 = 32 * g; c0 + 32 <= N; c0 += 32 * G) {
          uint32_t acc[32], h[16];
          chk_acc(p, c, static_cast<uint32_t>(s), tbase + static_cast<uint32_t>(c0), 32u);
          tmem_ld_x32(tbase + static_cast<uint32_t>(c0), acc);
          tmem_wait_ld();
          convert_pairs<V, 16, true>(acc, slope2, h);
          chk_a(p, c, static_cast<uint32_t>(s), a_tmem + static_cast<uint32_t>(c0 >> 1), 16u);
          tmem_st_x16(a_tmem + static_cast<uint32_t>(c0 >> 1), h);
        }
        if ((N & 31) && ((N >> 5) % G) == g) {
          const int c0 = N - 16;
          uint32_t acc[16], h[8];
          chk_acc(p, c, static_cast<uint32_t>(s), tbase + static_cast<uint32_t>(c0), 16u);
          tmem_ld_x16(tbase + static_cast<uint32_t>(c0), acc);
          tmem_wait_ld();
          convert_pairs<V, 8, true>(acc, slope2, h);
          chk_a(p, c, static_cast<uint32_t>(s), a_tmem + static_cast<uint32_t>(c0 >> 1), 8u);
          tmem_st_x8(a_tmem + static_cast<uint32_t>(c0 >> 1), h);
        }
        if (V == kVarRowMajor) rebuild_b(l + 1);
        tmem_wait_st();
      }
      tc_fence_before_sync();
      named_bar_sync(bar_id, bar_threads);
    }
    // Last layer: accumulator -> FP16 -> output staging -> TMA store.
    {
      const int l = L - 1;
      const uint32_t q = static_cast<uint32_t>(r * L + l);
      const int N = n_out;
      const uint32_t out_dst =
          c.sbase + p.sm_out +
          (static_cast<uint32_t>(s) * p.n_out_bufs + static_cast<uint32_t>(r) % p.n_out_bufs) *
              p.out_slot_bytes;
      // This staging buffer went to this warp's TMA stores n_out_bufs tiles
      // of this slot ago; they must have finished reading it.
      if (storer) {
        if (p.n_out_bufs > 1)
          bulk_wait_group_read<1>();
        else
          bulk_wait_group_read<0>();
      }
      __syncwarp();
      if (ok && has) ok = warp_wait(c.bar(kBarAccFull + s), q & 1u, p, c);
      if (ok && has) {
        tc_fence_after_sync();
        for (int c0 = 32 * g; c0 + 32 <= N; c0 += 32 * G) {
          uint32_t acc[32], h[16];
          chk_acc(p, c, static_cast<uint32_t>(s), tbase + static_cast<uint32_t>(c0), 32u);
          tmem_ld_x32(tbase + static_cast<uint32_t>(c0), acc);
          tmem_wait_ld();
          convert_pairs<V, 16, false>(acc, slope2, h);
          const uint32_t base = out_dst + out_chunk_off(c0);
#pragma unroll
          for (int cc = 0; cc < 4; ++cc) {
            chk_smem(p, c, base + swz(row * 64u + cc * 16u, 32), 16u);
            st_shared_v4_nc(base + swz(row * 64u + cc * 16u, 32), h[4 * cc], h[4 * cc + 1],
                            h[4 * cc + 2], h[4 * cc + 3]);
          }
        }
        if ((N & 31) && ((N >> 5) % G) == g) {
          const int c0 = N - 16;
          uint32_t acc[16], h[8];
          chk_acc(p, c, static_cast<uint32_t>(s), tbase + static_cast<uint32_t>(c0), 16u);
          tmem_ld_x16(tbase + static_cast<uint32_t>(c0), acc);
          tmem_wait_ld();
          convert_pairs<V, 8, false>(acc, slope2, h);
          const uint32_t base = out_dst + out_chunk_off(c0);
#pragma unroll
          for (int cc = 0; cc < 2; ++cc) {
            chk_smem(p, c, base + swz(row * 32u + cc * 16u, 16), 16u);
            st_shared_v4_nc(base + swz(row * 32u + cc * 16u, 16), h[4 * cc], h[4 * cc + 1],
                            h[4 * cc + 2], h[4 * cc + 3]);
          }
        }
        if (V == kVarRowMajor && (r + 1) * S + s < c.n_local) rebuild_b(0);
        fence_proxy_async_smem();  // staging tile -> TMA store (async proxy)
      }
      tc_fence_before_sync();
      named_bar_sync(bar_id, bar_threads);
      if (storer && ok && has) {
        const int64_t row0 = static_cast<int64_t>(t) * kTileM + quad * 32;
        if (row0 < p.n) {
          for (int c0 = 32 * g; c0 < N; c0 += 32 * G) {
            const int cols = (N - c0 >= 32) ? 32 : 16;
            tma_store_2d(&p.tm_out[swizzle_kind(cols)],
                         out_dst + out_chunk_off(c0) + static_cast<uint32_t>(quad * 32 * 2 * cols),
                         c0, static_cast<int32_t>(row0));
          }
        }
      }
      if (storer) bulk_commit_group();
    }
  }
  if (storer) bulk_wait_group_all();
}

// ------------------------------------------------------------------ streamed weights
// Networks whose packed weights do not fit next to the pipeline buffers
// stream them: lane 0 of the weight-producer warp copies each layer's
// K-segments -- each a contiguous N x 2w-byte piece of the packed image, at
// most 32 KB -- into a shared ring, in the order (round, layer, segment) in
// which every slot's issuing lane consumes them. A stage is released once
// every slot's MMAs on it have completed (or, for a slot with no tile in that
// round, once its lane has seen the stage).

__device__ __forceinline__ void run_weight_producer(const FusedParams& p, const Ctx& c) {
  const int32_t S = static_cast<int32_t>(p.n_slots);
  const int32_t n_rounds = (c.n_local + S - 1) / S;
  const uint32_t RW = p.n_wstages;
  bool ok = wait_phase(c.bar(kBarWLoad), 0, p.wait_ns, c.abort_flag, p.status);
  uint32_t g = 0;
  for (int32_t r = 0; r < n_rounds && ok; ++r) {
    for (int l = 0; l < p.L && ok; ++l) {
      const LayerRegs li = load_layer(p, c, l);
      for (int k = 0; k < li.K && ok;) {
        uint32_t off;
        int w, k0;
        locate(static_cast<uint32_t>(li.N), li.K, k, off, w, k0);
        const uint32_t st = g % RW;
        ok = wait_phase(c.bar(kBarWEmpty + st), ((g / RW) & 1u) ^ 1u, p.wait_ns, c.abort_flag,
                        p.status);
        if (!ok) break;
        const uint32_t bytes = static_cast<uint32_t>(li.N) * 2u * static_cast<uint32_t>(w);
        chk_smem(p, c, c.sbase + p.sm_wring + st * p.wstage_bytes, p.wstage_bytes);
        chk_fits(p, bytes, p.wstage_bytes);
        mbar_arrive_expect_tx(c.bar(kBarWFull + st), bytes);
        bulk_load(c.sbase + p.sm_wring + st * p.wstage_bytes, p.blob + li.w_off + off, bytes,
                  c.bar(kBarWFull + st));
        ++g;
        k = k0 + w;
      }
    }
  }
  // Drain: the last copies issued must land before the CTA may exit.
  const uint32_t first = g > RW ? g - RW : 0u;
  for (uint32_t gg = first; gg < g; ++gg)
    wait_drain(c.bar(kBarWFull + gg % RW), (gg / RW) & 1u, p.status);
}

template <int V>
__global__ void __launch_bounds__(is_stream(V) ? 32 * (16 + 2) : 32 * kMaxResidentWarps, 1)
    fused_mlp_kernel(const __grid_constant__ FusedParams p) {
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  const uint32_t raw = smem_u32(smem_raw);
  Ctx c;
  c.sbase = (raw + 1023u) & ~1023u;
  c.gbase = smem_raw + (c.sbase - raw);
  c.bars = c.sbase + p.sm_bar;
  c.abort_flag = reinterpret_cast<volatile uint32_t*>(c.gbase + p.sm_bar + kAbortOff);
  c.n_local = (static_cast<int32_t>(blockIdx.x) < p.num_tiles)
                  ? (p.num_tiles - static_cast<int32_t>(blockIdx.x) +
                     static_cast<int32_t>(gridDim.x) - 1) /
                        static_cast<int32_t>(gridDim.x)
                  : 0;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(c.gbase + p.sm_bar + kTmemSlotOff);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

  if (threadIdx.x == 0) {
    for (int s = 0; s < kMaxInStages; ++s) {
      mbar_init(c.bar(kBarInFull + s), 1);
      mbar_init(c.bar(kBarInEmpty + s), 1);
    }
    for (int s = 0; s < kMaxSlots; ++s) {
      mbar_init(c.bar(kBarAccFull + s), 1);
      mbar_init(c.bar(kBarDrain + s), 1);
    }
    for (int s = 0; s < kMaxBStages; ++s) mbar_init(c.bar(kBarBEmpty + s), 1);
    for (int s = 0; s < kMaxWStages; ++s) {
      mbar_init(c.bar(kBarWFull + s), 1);
      mbar_init(c.bar(kBarWEmpty + s), p.n_slots);
    }
    mbar_init(c.bar(kBarWLoad), 1);
    mbar_init(c.bar(kBarNever), 1);
    *c.abort_flag = 0u;
    fence_mbar_init();
  }
  if (warp == 0) {
    tmem_alloc(smem_u32(tmem_slot), p.tmem_cols);
    tmem_relinquish();
  }
  {
    // Ones tile (A of the layer-1 bias MMA) and the bias slabs (B of every
    // layer's bias MMA), 32-byte-swizzle K-major: row r's first 16-byte chunk
    // holds (value, 0 x 7) FP16, its second chunk zeros. Bias row j of the
    // concatenated biases is row j - bias_row0[l] of layer l's slab.
    const uint16_t* gb = reinterpret_cast<const uint16_t*>(p.blob + p.bias_off);
    const uint32_t total_rows = kTileM + p.n_bias;
    for (uint32_t idx = threadIdx.x; idx < 2u * total_rows; idx += blockDim.x) {
      const uint32_t rr = idx >> 1, ch = idx & 1u;
      uint32_t base, row, v;
      if (rr < kTileM) {
        base = c.sbase + p.sm_ones;
        row = rr;
        v = 0x3C00u;
      } else {
        const uint32_t j = rr - kTileM;
        int l = 0;
        while (l + 1 < p.L && j >= p.bias_row0[l + 1]) ++l;
        base = c.sbase + p.sm_bslab + p.bslab_off[l];
        row = j - p.bias_row0[l];
        v = gb[j];
      }
      chk_smem(p, c, base + swz(row * 32u + ch * 16u, 16), 16u);
      st_shared_v4(base + swz(row * 32u + ch * 16u, 16), ch ? 0u : v, 0u, 0u, 0u);
    }
    fence_proxy_async_smem();
  }
  tc_fence_before_sync();
  __syncthreads();
  tc_fence_after_sync();
  c.tmem = *tmem_slot;
  // The next dispatch of the stream may be scheduled now. It launches once
  // every CTA of this grid has executed this, that is once every one of them
  // is running and holds its tensor memory; its CTAs then take the SMs this
  // grid's CTAs leave and run their prologue while the last of them finish.
  // A CTA of the next grid that lands on an SM beside one of this grid can
  // therefore only ever wait for tensor memory that a running CTA of this
  // grid holds and will free: the waits cannot form a cycle.
  if (threadIdx.x == 0) griddep_launch_dependents();
  {
    // The constant A slab of every bias MMA: column 0 of every TMEM lane
    // holds (1.0, 0) as an FP16 pair, columns 1..7 zeros.
    if (warp < 4) {
      const uint32_t ones[8] = {0x3C00u, 0u, 0u, 0u, 0u, 0u, 0u, 0u};
      tmem_st_x8(c.tmem + (static_cast<uint32_t>(warp * 32) << 16) + p.ones_col, ones);
      tmem_wait_st();
    }
    tc_fence_before_sync();
    __syncthreads();
    tc_fence_after_sync();
  }

  if (warp == 0 && lane == 0) {
    // Stage the schedule (and the packed weight images) once for the whole
    // persistent loop.
    uint32_t wbytes = 0;  // resident weight images, if any
    if constexpr (V != kVarRowMajor && !is_stream(V)) wbytes = p.bias_off;
    mbar_arrive_expect_tx(c.bar(kBarWLoad), p.sched_bytes + wbytes);
    bulk_load(c.sbase + p.sm_sched, p.sched, p.sched_bytes, c.bar(kBarWLoad));
    for (uint32_t off = 0; off < wbytes; off += 32768u) {
      const uint32_t bytes = (wbytes - off) < 32768u ? (wbytes - off) : 32768u;
      bulk_load(c.sbase + p.sm_w + off, p.blob + off, bytes, c.bar(kBarWLoad));
    }
  }
  // Inputs, outputs and the status word may be shared with the previous
  // kernel of the stream: nothing below touches them before it completes.
  // The prologue above reads only the packed weights, which no kernel writes
  // except the packing kernel, and a dispatch that follows a packing kernel
  // is launched without programmatic serialisation.
  griddep_wait();
  if constexpr (is_stream(V)) {
    // Streamed weights: the slots' warps, then the weight producer, then the
    // input producer.
    const int slot_warps = 4 * static_cast<int>(p.n_slots * p.n_groups);
    if (warp < slot_warps) {
      run_slot<V>(p, c, warp, lane);
    } else if (warp == slot_warps) {
      if (lane == 0) run_weight_producer(p, c);
      __syncwarp();
    }
    if (warp == static_cast<int>(blockDim.x >> 5) - 1) {
      if (lane == 0) {
        run_input_producer(p, c);
        wait_drain(c.bar(kBarWLoad), 0, p.status);
      }
      __syncwarp();
    }
  } else {
    // Resident weights: the slots' issuing warps, the input producer, then
    // (from kEpiWarp0) the slots' epilogue warps.
    const int S = static_cast<int>(p.n_groups_issue);
    if (warp < S) {
      run_issuer<V>(p, c, warp, lane);
    } else if (warp == S) {
      if (lane == 0) {
        run_input_producer(p, c);
        wait_drain(c.bar(kBarWLoad), 0, p.status);
      }
      __syncwarp();
    } else if (warp >= kEpiWarp0) {
      run_epilogue<V>(p, c, warp - kEpiWarp0, lane);
    }
  }

  tc_fence_before_sync();
  __syncthreads();
  if (warp == 0) {
    tc_fence_after_sync();
    tmem_dealloc(c.tmem, p.tmem_cols);
  }
}

}  // namespace

// ------------------------------------------------------------------ host side
uint32_t build_schedule(const int32_t* dims, int L, const uint32_t* w_off, const uint32_t* rm_off,
                        Schedule& sc, uint32_t* bslab_bytes) {
  std::memset(&sc, 0, sizeof(sc));
  uint32_t boff = 0;
  for (int l = 0; l < L; ++l) {
    const int K = dims[l], N = dims[l + 1];
    LayerInfo& li = sc.layer[l];
    // Layer l's k-slabs start at row 16 l of the descriptor table, so the
    // kernel finds them without first reading the layer's entry.
    uint32_t slab = static_cast<uint32_t>(l) * 16u;
    li.K = K;
    li.N = N;
    li.slab_begin = slab;
    li.idesc = idesc_f16_f32(kTileM, static_cast<uint32_t>(N));
    li.bslab_off = boff;
    li.rm_off = rm_off[l];
    li.w_off = w_off[l];
    for (int k = 0; k < K; k += 16) {
      uint32_t aoff, boff_w;
      int w, k0;
      locate(kTileM, K, k, aoff, w, k0);
      locate(static_cast<uint32_t>(N), K, k, boff_w, w, k0);
      const uint32_t kb = static_cast<uint32_t>(k - k0) * 2u;
      const uint32_t sbo = 16u * static_cast<uint32_t>(w);
      sc.slab[slab].a = smem_desc(aoff + kb, sbo, swizzle_code(w));
      sc.slab[slab].b = smem_desc(boff_w + kb, sbo, swizzle_code(w));
      ++slab;
    }
    li.slab_end = slab;
    boff += align1024(static_cast<uint32_t>(N) * 32u);
  }
  *bslab_bytes = boff;
  return static_cast<uint32_t>(sizeof(LayerInfo) * kMaxLayers + sizeof(SlabDesc) * 16u * L);
}

uint32_t plan_fused_smem(FusedParams& p, const int32_t* dims, int variant, uint32_t smem_optin) {
  const int L = p.L;
  uint32_t nmax = 0, hmax = 16, bstage = 0, nb = 0;
  for (int l = 0; l < L; ++l) {
    const uint32_t N = static_cast<uint32_t>(dims[l + 1]);
    nmax = N > nmax ? N : nmax;
    if (l < L - 1 && N > hmax) hmax = N;
    const uint32_t ib = image_bytes(N, dims[l]);
    bstage = ib > bstage ? ib : bstage;
    nb += N;
  }
  p.n_bias = nb;
  p.d0 = dims[0];
  p.dL = dims[L];
  p.nslab_bits = 0;
  p.n16_bits = 0;
  for (int l = 0; l < L; ++l) {
    p.nslab_bits |= static_cast<uint64_t>((dims[l] >> 4) - 1) << (4 * l);
    p.n16_bits |= static_cast<uint64_t>((dims[l + 1] >> 4) - 1) << (4 * l);
  }
  const uint32_t acc_cols = (nmax + 31u) & ~31u;  // widest layer, a multiple of 32
  // output staging: 8 KB per 32-column chunk, 4 KB for a trailing 16-column one
  p.out_slot_bytes = static_cast<uint32_t>(p.dL >> 5) * (kTileM * 64u) +
                     ((p.dL & 31) ? kTileM * 32u : 0u);
  p.b_stage_bytes = (variant == kVarRowMajor) ? align1024(bstage) : 0u;
  const uint32_t stage = align1024(image_bytes(kTileM, p.d0));
  // Streamed weights: a ring of stages, each one K-segment of one layer.
  uint32_t wseg = 0;
  for (int l = 0; l < L; ++l) {
    const uint32_t wmax = dims[l] >= 64 ? 64u : (dims[l] >= 32 ? 32u : 16u);
    const uint32_t b = static_cast<uint32_t>(dims[l + 1]) * 2u * wmax;
    wseg = b > wseg ? b : wseg;
  }
  wseg = align1024(wseg);

  // Resident weights first: the most tile slots TMEM allows (up to 5; per
  // slot the accumulator and the A region, plus one shared 32-column block
  // for the ones slab), two input stages per slot before one, two output
  // buffers before one. If the weights do not fit (fused and
  // scalar-activation variants), stream them with at most 3 slots and the
  // deepest weight ring (4 down to 2 stages) that fits.
  // The narrow-precision variant: streamed weights only, on networks that
  // have E4M3 images; its A region holds four E4M3 values per column.
  const bool fp8 = variant == kVarFp8;
  if (fp8) {
    if (L < 2) return 0;
    for (int l = 1; l < L; ++l)
      if (dims[l] % 32 != 0) return 0;
  }
  for (int mode = fp8 ? 1 : 0; mode < 2; ++mode) {
    const bool streamed = mode == 1;
    if (streamed && variant == kVarRowMajor) break;
    p.a_col = acc_cols;
    const uint32_t max_slots = streamed ? static_cast<uint32_t>(kStreamSlots) : static_cast<uint32_t>(kMaxSlots);
    for (uint32_t slots = max_slots; slots >= 1; --slots) {
      // A wholly in TMEM; or, for streamed FP16 weights (fused kernel) when
      // that leaves too few slots, its first a_tmem_k columns (a multiple of
      // 64) in TMEM and the rest in shared memory, if every hidden width
      // above a_tmem_k is a multiple of 64 (whole 64-column segments).
      p.a_tmem_k = hmax;
      p.slot_cols = acc_cols + (((hmax / (fp8 ? 4u : 2u)) + 31u) & ~31u);
      if (slots * p.slot_cols + 32u > 512u && streamed &&
          (variant == kVarFused || variant == kVarPaired)) {
        const uint32_t room = (512u - 32u) / slots;
        const uint32_t k = room > acc_cols ? ((room - acc_cols) * 2u) & ~63u : 0u;
        bool ok = k >= 64u;
        for (int l = 1; l < L && ok; ++l)
          if (static_cast<uint32_t>(dims[l]) > k && dims[l] % 64 != 0) ok = false;
        if (!ok) continue;
        p.a_tmem_k = k;
        p.slot_cols = acc_cols + k / 2u;
      }
      p.a_smem_bytes = hmax > p.a_tmem_k ? kTileM * 2u * (hmax - p.a_tmem_k) : 0u;
      const uint32_t used = slots * p.slot_cols + 32u;
      if (used > 512u) continue;
      const uint32_t groups = slots >= 3 ? 1u : 4u / slots;
      p.n_b_stages = (variant == kVarRowMajor) ? slots : 0u;
      for (uint32_t wst = streamed ? kMaxWStages : 0u; wst >= (streamed ? 2u : 0u); --wst) {
        for (uint32_t depth = 2; depth >= 1; --depth) {
          for (uint32_t obufs = kOutBufs; obufs >= 1; --obufs) {
            uint32_t off = 0;
            p.sm_w = 0;
            off += (variant == kVarRowMajor || streamed) ? 0u : align1024(p.bias_off);
            p.sm_sched = off;
            off += align1024(p.sched_bytes);
            p.sm_bslab = off;
            off += align1024(p.bslab_bytes);
            p.sm_ones = off;
            off += kOnesTileBytes;
            p.sm_out = off;
            off += slots * obufs * p.out_slot_bytes;
            p.sm_b = off;
            off += p.n_b_stages * p.b_stage_bytes;
            p.sm_wring = off;
            off += wst * wseg;
            p.sm_bar = off;
            off += 1024u;  // barrier block, keeps the input ring 1024-aligned
            p.sm_in = off;
            off += slots * depth * stage;
            p.sm_a = off;
            off += slots * p.a_smem_bytes;
            const uint32_t total = off + 1024u;  // + alignment slack of the dynamic smem base
            if (total <= smem_optin) {
              uint32_t cols = 32;
              while (cols < used) cols <<= 1;
              p.tmem_cols = cols;
              p.chk_tmem_cols = used;
              p.smem_end = off;
              p.ones_col = slots * p.slot_cols;
              p.n_slots = slots;
              // Issue groups: one tile region each, or (paired-tiles variant,
              // one column group per warp) pairs of regions while at least two
              // are left.
              {
                const bool pair = variant == kVarPaired && !streamed && groups == 1;
                uint32_t ng = 0;
                for (uint32_t r0 = 0; r0 < slots;) {
                  const uint32_t t = (pair && slots - r0 >= 2) ? 2u : 1u;
                  p.grp_first[ng] = r0;
                  p.grp_tiles[ng] = t;
                  for (uint32_t k = 0; k < t; ++k) p.grp_of[r0 + k] = ng;
                  r0 += t;
                  ++ng;
                }
                p.n_groups_issue = ng;
              }
              p.n_groups = groups;
              p.n_threads = streamed ? 32u * (4u * slots * groups + 2u)
                                     : 32u * (static_cast<uint32_t>(kEpiWarp0) + 4u * slots * groups);
              p.in_stage_bytes = stage;
              p.n_in_stages = depth;
              p.n_out_bufs = obufs;
              p.stream_w = streamed ? 1u : 0u;
              p.n_wstages = wst;
              p.wstage_bytes = wseg;
              return total;
            }
          }
        }
        if (!streamed) break;
      }
    }
  }
  return 0;
}

// The opt-in shared-memory limit of a kernel instantiation is a property of
// the function in one device's context: it is set once per device (the
// device current at launch), under a lock so that host threads launching
// concurrently do not race on it.
constexpr int kMaxDevices = 64;

template <int V>
static cudaError_t configure_for_device() {
  static std::atomic<bool> done[kMaxDevices];
  static std::mutex mu;
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
  if (done[dev].load(std::memory_order_acquire)) return cudaSuccess;
  std::lock_guard<std::mutex> lk(mu);
  if (done[dev].load(std::memory_order_relaxed)) return cudaSuccess;
  int optin = 0;
  e = cudaDeviceGetAttribute(&optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev);
  if (e == cudaSuccess)
    e = cudaFuncSetAttribute(fused_mlp_kernel<V>, cudaFuncAttributeMaxDynamicSharedMemorySize, optin);
  if (e == cudaSuccess) done[dev].store(true, std::memory_order_release);
  return e;
}

template <int V>
static cudaError_t launch_variant(const FusedParams& p, int grid, uint32_t smem, cudaStream_t stream,
                                  bool overlap) {
  const cudaError_t e = configure_for_device<V>();
  if (e != cudaSuccess) return e;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>(grid));
  cfg.blockDim = dim3(p.n_threads);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = overlap ? 1 : 0;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, fused_mlp_kernel<V>, p);
}

cudaError_t launch_fused(const FusedParams& p, int variant, int grid, uint32_t smem,
                         cudaStream_t stream, bool overlap) {
  if (p.stream_w) {
    if (variant == kVarFused || variant == kVarPaired)
      return p.a_smem_bytes ? launch_variant<kVarFusedStreamSplitA>(p, grid, smem, stream, overlap)
                            : launch_variant<kVarFusedStream>(p, grid, smem, stream, overlap);
    if (variant == kVarScalar) return launch_variant<kVarScalarStream>(p, grid, smem, stream, overlap);
    if (variant == kVarFp8) return launch_variant<kVarFp8Stream>(p, grid, smem, stream, overlap);
    return cudaErrorInvalidValue;
  }
  switch (variant) {
    case kVarFused:
    case kVarPaired: return launch_variant<kVarFused>(p, grid, smem, stream, overlap);
    case kVarRowMajor: return launch_variant<kVarRowMajor>(p, grid, smem, stream, overlap);
    case kVarScalar: return launch_variant<kVarScalar>(p, grid, smem, stream, overlap);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace nm
