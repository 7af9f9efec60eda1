// nm_fused.cu -- persistent fused inference kernel of the FP16 MLP on sm_103a.
//
// One CTA per SM walks 128-sample tiles t = blockIdx.x, blockIdx.x + grid, ...
// and runs every layer of the network on each tile without leaving the SM
// ("Optimization Techniques: Squeezing the Silicon", "Kernel Fusion": one
// write to memory, intermediates stay on chip). Roles, by warp:
//   warp 0      producer: TMA loads of the [128 x d0] input tiles into a ring
//               (and, in the row-major ablation, rebuilds every layer's B
//               operand from the row-major weights for every tile);
//   warp 1      one thread issues the tcgen05.mma chain of each layer,
//               D[128 x N] (FP32, TMEM) = A[128 x K] (FP16, smem) * W^T;
//   warps 2..5  epilogue: tcgen05.ld of the accumulator rows, FP32 bias add,
//               FP16 rounding, FP16 activation max(h, h*half(0.01)), and a
//               16-byte store into the next layer's A tile (or into the
//               output staging tile, which leaves by TMA store).
// Two tiles are in flight (two TMEM accumulator slots, two activation tiles)
// so one tile's epilogue overlaps the other tile's MMAs.
//
// The page "Profiling neural material inference" fixes the arithmetic
// ("Experiment setup": the full layer chain per evaluation; "Bad versus good
// activation": the FP16 max form) and supplies the two ablations compiled
// here as variants: "Row-major versus InferencingOptimal weights" (B operand
// rebuilt from row-major memory per tile) and the indexed-lane activation.
//
// Every wait is bounded by a wall-clock limit. A wait that gives up sets the
// device status word and a CTA-wide abort flag; every role then stops, waits
// (with a fixed limit) for its own copies and MMAs in flight, and the CTA
// frees its tensor memory and exits.
#include <cuda_fp16.h>

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
  __device__ __forceinline__ uint32_t bar(int i) const {
    return bars + static_cast<uint32_t>(i) * 8u;
  }
};

// Bounded wait on an mbarrier phase. Gives up (and raises the abort flag and
// the status word) when `limit_ns` passes or another role has given up.
__device__ __noinline__ bool wait_phase(uint32_t bar, uint32_t parity, uint64_t limit_ns,
                                        volatile uint32_t* abort_flag, uint32_t* status) {
  if (mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = globaltimer_ns();
  uint32_t spins = 0;
  while (true) {
    if (mbar_try_wait(bar, parity)) return true;
    if (*abort_flag) return false;
    if ((++spins & 63u) == 0u && globaltimer_ns() - t0 > limit_ns) {
      *abort_flag = 1u;
      atomicOr(status, kStatusTimeout);
      return false;
    }
  }
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

// FP32 accumulator pair + FP32 bias pair -> FP16 pair (round to nearest even),
// then the activation when `act` is set. Column 2j goes to the low half.
template <int V>
__device__ __forceinline__ void epilogue_chunk(const uint32_t* acc, const float* bias, int npairs,
                                               bool act, __half2 slope2, uint32_t* out) {
#pragma unroll
  for (int j = 0; j < 16; ++j) {
    if (j < npairs) {
      const float2 a = make_float2(__uint_as_float(acc[2 * j]), __uint_as_float(acc[2 * j + 1]));
      const float2 b = *reinterpret_cast<const float2*>(bias + 2 * j);
      const float2 v = __fadd2_rn(a, b);
      __half2 h = __float22half2_rn(v);
      if (V != kVarScalar) {
        if (act) h = __hmax2(h, __hmul2(h, slope2));
      }
      out[j] = *reinterpret_cast<uint32_t*>(&h);
    }
  }
  if (V == kVarScalar && act) {
    // The page's indexed-lane form: every FP16 value visited one by one with
    // a dynamic index and a branch.
    __half lanes[32];
#pragma unroll
    for (int j = 0; j < 16; ++j) {
      __half2 h = *reinterpret_cast<__half2*>(&out[j]);
      lanes[2 * j] = __low2half(h);
      lanes[2 * j + 1] = __high2half(h);
    }
    const __half slope = __low2half(slope2);
    const __half zero = __float2half_rn(0.0f);
#pragma unroll 1
    for (int e = 0; e < 2 * npairs; ++e) {
      if (__hlt(lanes[e], zero)) lanes[e] = __hmul(lanes[e], slope);
    }
#pragma unroll
    for (int j = 0; j < 16; ++j) {
      __half2 h = __halves2half2(lanes[2 * j], lanes[2 * j + 1]);
      out[j] = *reinterpret_cast<uint32_t*>(&h);
    }
  }
}

__device__ __forceinline__ void issue_input_tma(const FusedParams& p, uint32_t dst, uint32_t bar,
                                                int32_t tile) {
  const int K = p.dims[0];
  for (int k = 0; k < K;) {
    uint32_t off;
    int w, k0;
    locate(kTileM, K, k, off, w, k0);
    tma_load_2d(dst + off, &p.tm_in[swizzle_kind(w)], bar, k0, tile * kTileM);
    k = k0 + w;
  }
}

// ------------------------------------------------------------------ producer
template <int V>
__device__ __forceinline__ void run_producer(const FusedParams& p, const Ctx& c, int lane) {
  const uint32_t R = p.n_in_stages;
  int32_t last_round[kMaxInStages];
#pragma unroll
  for (int s = 0; s < kMaxInStages; ++s) last_round[s] = -1;

  uint32_t i = 0, g = 0;
  bool ok = true;
  for (int32_t t = blockIdx.x; t < p.num_tiles && ok; t += gridDim.x, ++i) {
    const uint32_t st = i % R, rnd = i / R;
    if (lane == 0) {
      ok = wait_phase(c.bar(kBarInEmpty + st), (rnd & 1u) ^ 1u, p.wait_ns, c.abort_flag, p.status);
      if (ok) {
        mbar_arrive_expect_tx(c.bar(kBarInFull + st), static_cast<uint32_t>(kTileM * 2 * p.dims[0]));
        issue_input_tma(p, c.sbase + p.sm_in + st * p.in_stage_bytes, c.bar(kBarInFull + st), t);
        last_round[st] = static_cast<int32_t>(rnd);
      }
    }
    if (V == kVarRowMajor) {
      ok = __shfl_sync(0xFFFFFFFFu, ok, 0);
      // Rebuild every layer's B operand for this tile from the row-major
      // weights: 16-byte row-major loads, swizzled 16-byte smem stores.
      for (int l = 0; l < p.L && ok; ++l, ++g) {
        const uint32_t bs = g % p.n_b_stages, brnd = g / p.n_b_stages;
        const bool got = wait_phase(c.bar(kBarBEmpty + bs), (brnd & 1u) ^ 1u, p.wait_ns,
                                    c.abort_flag, p.status);
        ok = __all_sync(0xFFFFFFFFu, got);
        if (!ok) break;
        const int K = p.dims[l], N = p.dims[l + 1], kc = K >> 3;
        const uint16_t* Wl = p.mirror + p.rm_off[l];
        const uint32_t stage = c.sbase + p.sm_b + bs * p.b_stage_bytes;
        for (int idx = lane; idx < N * kc; idx += 32) {
          const int n = idx / kc, col = (idx - n * kc) << 3;
          const uint4 v = __ldg(reinterpret_cast<const uint4*>(Wl + n * K + col));
          uint32_t off;
          int w, k0;
          locate(static_cast<uint32_t>(N), K, col, off, w, k0);
          st_shared_v4(stage + off + swz(static_cast<uint32_t>(n * 2 * w + (col - k0) * 2), w),
                       v.x, v.y, v.z, v.w);
        }
        fence_proxy_async_smem();
        mbar_arrive(c.bar(kBarBFull + bs));
      }
    }
  }
  if (lane == 0) {
    // Drain: every copy this warp issued (input tiles, and the one-time
    // weight staging) must land before the CTA may exit.
    for (uint32_t s = 0; s < R; ++s)
      if (last_round[s] >= 0) wait_drain(c.bar(kBarInFull + s), last_round[s] & 1, p.status);
    if (V != kVarRowMajor) wait_drain(c.bar(kBarWLoad), 0, p.status);
  }
}

// ------------------------------------------------------------------ MMA issuer
template <int V>
__device__ __forceinline__ void run_mma(const FusedParams& p, const Ctx& c) {
  const uint32_t R = p.n_in_stages;
  const int L = p.L;
  bool ok = true;
  if (p.test_stall) ok = wait_phase(c.bar(kBarNever), 0, p.wait_ns, c.abort_flag, p.status);
  if (ok && V != kVarRowMajor)
    ok = wait_phase(c.bar(kBarWLoad), 0, p.wait_ns, c.abort_flag, p.status);
  uint32_t i = 0, g = 0;
  for (int32_t t = blockIdx.x; t < p.num_tiles && ok; t += gridDim.x, ++i) {
    const uint32_t s = i & 1u, st = i % R, rnd = i / R;
    const uint32_t d_tmem = c.tmem + s * p.nmax;
    for (int l = 0; l < L; ++l) {
      const int q = static_cast<int>((i >> 1) * L + l) - 1;
      if (q >= 0 && !wait_phase(c.bar(kBarActReady + s), q & 1, p.wait_ns, c.abort_flag, p.status)) {
        ok = false;
        break;
      }
      if (l == 0 &&
          !wait_phase(c.bar(kBarInFull + st), rnd & 1u, p.wait_ns, c.abort_flag, p.status)) {
        ok = false;
        break;
      }
      uint32_t b_base, bs = 0;
      if (V == kVarRowMajor) {
        bs = g % p.n_b_stages;
        if (!wait_phase(c.bar(kBarBFull + bs), (g / p.n_b_stages) & 1u, p.wait_ns, c.abort_flag,
                        p.status)) {
          ok = false;
          break;
        }
        b_base = c.sbase + p.sm_b + bs * p.b_stage_bytes;
      } else {
        b_base = c.sbase + p.sm_w + p.w_off[l];
      }
      tc_fence_after_sync();
      const uint32_t a_base = (l == 0) ? (c.sbase + p.sm_in + st * p.in_stage_bytes)
                                       : (c.sbase + p.sm_act + s * p.act_slot_bytes);
      const int K = p.dims[l], N = p.dims[l + 1];
      const uint32_t idesc = idesc_f16_f32(kTileM, static_cast<uint32_t>(N));
      for (int k = 0; k < K; k += 16) {
        uint32_t aoff, boff;
        int w, k0;
        locate(kTileM, K, k, aoff, w, k0);
        locate(static_cast<uint32_t>(N), K, k, boff, w, k0);
        const uint32_t kb = static_cast<uint32_t>(k - k0) * 2u;
        const uint32_t sbo = 16u * static_cast<uint32_t>(w);
        const uint64_t adesc = smem_desc(a_base + aoff + kb, sbo, swizzle_code(w));
        const uint64_t bdesc = smem_desc(b_base + boff + kb, sbo, swizzle_code(w));
        umma_f16_ss(d_tmem, adesc, bdesc, idesc, k > 0 ? 1u : 0u);
      }
      umma_commit(c.bar(kBarAccFull + s));
      if (l == 0) umma_commit(c.bar(kBarInEmpty + st));
      if (V == kVarRowMajor) {
        umma_commit(c.bar(kBarBEmpty + bs));
        ++g;
      }
    }
  }
  // Drain: all MMAs issued by this thread complete before teardown.
  umma_commit(c.bar(kBarDrain));
  wait_drain(c.bar(kBarDrain), 0, p.status);
}

// ------------------------------------------------------------------ epilogue
template <int V>
__device__ __forceinline__ void run_epilogue(const FusedParams& p, const Ctx& c, int warp,
                                             int lane) {
  const int quad = warp & 3;  // TMEM lane quadrant this warp may access
  const uint32_t row = static_cast<uint32_t>(quad * 32 + lane);
  const uint32_t lane_bits = static_cast<uint32_t>(quad * 32) << 16;
  const __half2 slope2 = __float2half2_rn(0.01f);  // half(0.01)
  const float* sbias = reinterpret_cast<const float*>(c.gbase + p.sm_bias);
  const int L = p.L;
  uint32_t i = 0;
  for (int32_t t = blockIdx.x; t < p.num_tiles; t += gridDim.x, ++i) {
    const uint32_t s = i & 1u;
    bool ok = true;
    for (int l = 0; l < L; ++l) {
      const uint32_t q = (i >> 1) * static_cast<uint32_t>(L) + static_cast<uint32_t>(l);
      // All lanes poll; the warp proceeds only together (the TMEM loads below
      // are warp-collective).
      const bool got = wait_phase(c.bar(kBarAccFull + s), q & 1u, p.wait_ns, c.abort_flag, p.status);
      if (!__all_sync(0xFFFFFFFFu, got)) {
        ok = false;
        break;
      }
      tc_fence_after_sync();
      const int N = p.dims[l + 1];
      const bool last = (l == L - 1);
      const float* bias = sbias + p.bias_f_off[l];
      const uint32_t dst = last ? (c.sbase + p.sm_out + s * p.out_slot_bytes)
                                : (c.sbase + p.sm_act + s * p.act_slot_bytes);
      if (last) {
        // The staging tile of slot s was last handed to a TMA store kSlots
        // tiles ago; make sure that store has finished reading it.
        if (lane == 0) bulk_wait_group_read<kSlots - 1>();
        __syncwarp();
      }
      const uint32_t tbase = c.tmem + lane_bits + s * p.nmax;
      for (int c0 = 0; c0 < N; c0 += 32) {
        uint32_t acc[32];
        uint32_t h[16];
        const int cols = (N - c0 >= 32) ? 32 : 16;
        if (cols == 32) {
          tmem_ld_x32(tbase + static_cast<uint32_t>(c0), acc);
        } else {
          tmem_ld_x16(tbase + static_cast<uint32_t>(c0), *reinterpret_cast<uint32_t(*)[16]>(acc));
        }
        tmem_wait_ld();
        epilogue_chunk<V>(acc, bias + c0, cols >> 1, !last, slope2, h);
#pragma unroll
        for (int cc = 0; cc < 4; ++cc) {
          if (cc * 8 < cols) {
            const int col = c0 + cc * 8;
            uint32_t off;
            int w, k0;
            locate(kTileM, N, col, off, w, k0);
            const uint32_t lin = row * 2u * static_cast<uint32_t>(w) + static_cast<uint32_t>(col - k0) * 2u;
            st_shared_v4(dst + off + swz(lin, w), h[4 * cc], h[4 * cc + 1], h[4 * cc + 2],
                         h[4 * cc + 3]);
          }
        }
      }
      tc_fence_before_sync();
      fence_proxy_async_smem();
      mbar_arrive(c.bar(kBarActReady + s));
      if (last) {
        __syncwarp();
        if (lane == 0) {
          const int64_t row0 = static_cast<int64_t>(t) * kTileM + quad * 32;
          if (row0 < p.n) {
            for (int k = 0; k < N;) {
              uint32_t off;
              int w, k0;
              locate(kTileM, N, k, off, w, k0);
              tma_store_2d(&p.tm_out[swizzle_kind(w)],
                           dst + off + static_cast<uint32_t>(quad * 32) * 2u * static_cast<uint32_t>(w),
                           k0, static_cast<int32_t>(row0));
              k = k0 + w;
            }
          }
          bulk_commit_group();
        }
      }
    }
    if (!ok) break;
  }
  if (lane == 0) bulk_wait_group_all();
}

template <int V>
__global__ void __launch_bounds__(kFusedThreads, 1)
    fused_mlp_kernel(const __grid_constant__ FusedParams p) {
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  const uint32_t raw = smem_u32(smem_raw);
  Ctx c;
  c.sbase = (raw + 1023u) & ~1023u;
  c.gbase = smem_raw + (c.sbase - raw);
  c.bars = c.sbase + p.sm_bar;
  c.abort_flag = reinterpret_cast<volatile uint32_t*>(c.gbase + p.sm_bar + kAbortOff);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(c.gbase + p.sm_bar + kTmemSlotOff);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

  if (threadIdx.x == 0) {
    for (int s = 0; s < kMaxInStages; ++s) {
      mbar_init(c.bar(kBarInFull + s), 1);
      mbar_init(c.bar(kBarInEmpty + s), 1);
    }
    for (int s = 0; s < kSlots; ++s) {
      mbar_init(c.bar(kBarAccFull + s), 1);
      mbar_init(c.bar(kBarActReady + s), 128);
    }
    for (int s = 0; s < kMaxBStages; ++s) {
      mbar_init(c.bar(kBarBFull + s), 32);
      mbar_init(c.bar(kBarBEmpty + s), 1);
    }
    mbar_init(c.bar(kBarWLoad), 1);
    mbar_init(c.bar(kBarDrain), 1);
    mbar_init(c.bar(kBarNever), 1);
    *c.abort_flag = 0u;
    fence_mbar_init();
  }
  if (warp == 0) {
    tmem_alloc(smem_u32(tmem_slot), p.tmem_cols);
    tmem_relinquish();
  }
  {
    // FP16 biases of every layer -> FP32 in shared memory (exact widening).
    float* sbias = reinterpret_cast<float*>(c.gbase + p.sm_bias);
    const __half* gb = reinterpret_cast<const __half*>(p.blob + p.bias_off);
    for (uint32_t j = threadIdx.x; j < p.n_bias; j += kFusedThreads) sbias[j] = __half2float(gb[j]);
  }
  tc_fence_before_sync();
  __syncthreads();
  tc_fence_after_sync();
  c.tmem = *tmem_slot;

  if (warp == 0) {
    if (V != kVarRowMajor && lane == 0) {
      // Stage the packed weight images once for the whole persistent loop.
      mbar_arrive_expect_tx(c.bar(kBarWLoad), p.bias_off);
      for (uint32_t off = 0; off < p.bias_off; off += 32768u) {
        const uint32_t bytes = (p.bias_off - off) < 32768u ? (p.bias_off - off) : 32768u;
        bulk_load(c.sbase + p.sm_w + off, p.blob + off, bytes, c.bar(kBarWLoad));
      }
    }
    if (V == kVarRowMajor || lane == 0) run_producer<V>(p, c, lane);
  } else if (warp == 1) {
    if (lane == 0) run_mma<V>(p, c);
    __syncwarp();
  } else {
    run_epilogue<V>(p, c, warp, lane);
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
uint32_t plan_fused_smem(FusedParams& p, int variant, uint32_t smem_optin) {
  const int L = p.L;
  uint32_t nmax = 0, act_w = 16, bstage = 0, nb = 0;
  for (int l = 0; l < L; ++l) {
    const uint32_t N = static_cast<uint32_t>(p.dims[l + 1]);
    nmax = N > nmax ? N : nmax;
    if (l < L - 1 && N > act_w) act_w = N;
    const uint32_t ib = image_bytes(N, p.dims[l]);
    bstage = ib > bstage ? ib : bstage;
    p.bias_f_off[l] = nb;
    nb += N;
  }
  p.n_bias = nb;
  // TMEM columns per tile slot: the widest layer, rounded up to a power of two.
  uint32_t slot = 32;
  while (slot < nmax) slot <<= 1;
  p.nmax = slot;
  uint32_t cols = 32;
  while (cols < kSlots * slot) cols <<= 1;
  if (cols > 512) return 0;
  p.tmem_cols = cols;

  p.in_stage_bytes = image_bytes(kTileM, p.dims[0]);
  p.act_slot_bytes = align1024(image_bytes(kTileM, static_cast<int>(act_w)));
  p.out_slot_bytes = align1024(image_bytes(kTileM, p.dims[L]));
  p.b_stage_bytes = (variant == kVarRowMajor) ? align1024(bstage) : 0u;
  p.n_b_stages = (variant == kVarRowMajor) ? kMaxBStages : 0u;

  uint32_t off = 0;
  p.sm_w = 0;
  off += (variant == kVarRowMajor) ? 0u : align1024(p.bias_off);
  p.sm_bias = off;
  off += align1024(nb * 4u);
  p.sm_act = off;
  off += kSlots * p.act_slot_bytes;
  p.sm_out = off;
  off += kSlots * p.out_slot_bytes;
  p.sm_b = off;
  off += p.n_b_stages * p.b_stage_bytes;
  p.sm_bar = off;
  off += 1024u;  // barrier block (256 B used), keeps the input ring 1024-aligned
  p.sm_in = off;
  const uint32_t fixed = off + 1024u;  // + alignment slack of the dynamic smem base
  int stages = kMaxInStages;
  while (stages >= 2 && fixed + static_cast<uint32_t>(stages) * align1024(p.in_stage_bytes) > smem_optin)
    --stages;
  if (stages < 2) return 0;
  p.in_stage_bytes = align1024(p.in_stage_bytes);
  p.n_in_stages = static_cast<uint32_t>(stages);
  return fixed + static_cast<uint32_t>(stages) * p.in_stage_bytes;
}

template <int V>
static cudaError_t launch_variant(const FusedParams& p, int grid, uint32_t smem, cudaStream_t stream) {
  static bool configured = false;
  if (!configured) {
    cudaError_t e = cudaFuncSetAttribute(fused_mlp_kernel<V>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, 232448);
    if (e != cudaSuccess) return e;
    configured = true;
  }
  fused_mlp_kernel<V><<<grid, kFusedThreads, smem, stream>>>(p);
  return cudaGetLastError();
}

cudaError_t launch_fused(const FusedParams& p, int variant, int grid, uint32_t smem,
                         cudaStream_t stream) {
  switch (variant) {
    case kVarFused: return launch_variant<kVarFused>(p, grid, smem, stream);
    case kVarRowMajor: return launch_variant<kVarRowMajor>(p, grid, smem, stream);
    case kVarScalar: return launch_variant<kVarScalar>(p, grid, smem, stream);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace nm
