/*
 * nm_mlp.h -- C ABI of libnmmlp: batched inference of a small fused FP16 MLP
 * on one NVIDIA GB300 (sm_103a).
 *
 * The problem statement these calls follow comes from the page "Profiling
 * neural material inference":
 *  - "Experiment setup": one dispatch evaluates a batch of inputs, each
 *    through the complete eight-affine-layer network (E1/E2/E3/F/S/D/H/O);
 *    the timing covers the whole inference pass.
 *  - "Bad versus good activation": between layers the FP16 activation
 *    value = max(value, value * half(0.01)) is applied to the whole vector.
 *  - "Row-major versus InferencingOptimal weights": the network's canonical
 *    weights are FP16 row-major matrices; before inference they are converted
 *    once into an opaque, device-dependent layout whose size the application
 *    queries; the conversion changes neither the network nor the activation
 *    and is paid only when the weights change.
 * and from "Working with Cooperative Matrices", "Hardware Constraints and
 * Capabilities": FP16 operands with FP32 accumulation, and 16-byte aligned
 * addresses for every load and store of matrix data.
 *
 * Arithmetic of one evaluation (layer l = 0..L-1, K = d_l, N = d_{l+1}):
 *   acc[o] = sum_k x[k] * W_l[o][k]          FP16 x FP16 products, FP32 sum
 *   v[o]   = acc[o] + b_l[o]                  FP32
 *   h[o]   = fp16_rn(v[o])                    round to nearest even
 *   h[o]   = max(h[o], h[o] * half(0.01))     FP16, for every layer but the last
 * The tensor cores sum the K products in an order and with an internal
 * precision of their own, so results match a k-ordered FP32 sum to within
 * |gpu - cpu| <= 1e-2 + 1e-2 |cpu| per element, and bit for bit wherever
 * every partial sum is exact in FP32.
 *
 * Conventions for every call:
 *  - Device pointers are CUDA device addresses on the device that was current
 *    when nm_mlp_create ran; that device must be current for every later call.
 *  - Every matrix pointer must be 16-byte aligned; matrices are row-major and
 *    tightly packed (row stride = width * 2 bytes).
 *  - nm_mlp_pack_weights, nm_mlp_unpack_weights and nm_mlp_infer are
 *    stream-ordered and asynchronous: they enqueue work on `stream` and return;
 *    the caller keeps the buffers alive until the stream has passed the call.
 *    A NULL stream is the legacy default stream.
 *  - A handle is not thread-safe. Infers on different streams may overlap if
 *    their outputs do not.
 *  - Errors are returned, never printed or raised. Argument errors are found
 *    on the host before anything is enqueued.
 */
#ifndef NM_MLP_H
#define NM_MLP_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* A CUDA stream (the same object as cudaStream_t / CUstream). */
typedef struct CUstream_st *nm_stream;

/* Opaque network handle: layer dims, the packed weight blob in device memory
 * and a device status word. */
typedef struct nm_mlp nm_mlp;

typedef enum nm_status {
    NM_OK = 0,
    NM_ERR_INVALID_ARG = 1,  /* NULL / misaligned pointer, negative n, bad dims array */
    NM_ERR_UNSUPPORTED = 2,  /* dims outside the supported set, or not an sm_103 device */
    NM_ERR_NOT_PACKED = 3,   /* infer or unpack before nm_mlp_pack_weights */
    NM_ERR_OOM = 4,          /* device allocation failed */
    NM_ERR_CUDA = 5,         /* a CUDA runtime/driver call or launch failed */
    NM_ERR_TIMEOUT = 6,      /* a bounded wait inside a kernel gave up (see nm_mlp_device_status) */
    NM_ERR_RANGE_CHECK = 7   /* checking build only: a kernel-side range check failed */
} nm_status;

/* Kernel variants. NM_VARIANT_FUSED is the product path; the row-major and
 * scalar-activation variants are the page's two performance cliffs, kept as
 * measured ablations; the paired-tiles variant is a measured alternative
 * schedule. Those four produce bit-identical outputs. The narrow-precision
 * variant computes differently (see its entry). */
typedef enum nm_variant {
    /* Packed weights staged once per CTA into shared memory; packed half2
     * activation ("Row-major versus InferencingOptimal weights", optimal
     * layout; "Bad versus good activation", good form). */
    NM_VARIANT_FUSED = 0,
    /* Ablation of the weight layout: for every 128-sample tile and every
     * layer the B operand is rebuilt in shared memory from the row-major
     * weights in global memory instead of being staged once packed
     * ("Row-major versus InferencingOptimal weights", row-major side). */
    NM_VARIANT_ROWMAJOR_WEIGHTS = 1,
    /* Ablation of the activation: the epilogue walks the FP16 values one by
     * one with a dynamic index and a branch, if (h < 0) h *= half(0.01)
     * ("Bad versus good activation", bad form). */
    NM_VARIANT_SCALAR_ACTIVATION = 2,
    /* The fused kernel with two tile regions (256 samples) per issuing warp:
     * one warp issues both tiles' MMA chains of a layer and meets both
     * tiles' epilogue warps at one barrier (five regions are issued as
     * 2 + 2 + 1). A larger M per issue than the default one tile per
     * issuing warp; measured slower on the benchmark networks, kept as a
     * measured alternative. Same arithmetic, bit-identical outputs. */
    NM_VARIANT_PAIRED_TILES = 3,
    /* Narrow-precision weights ("Optimization Techniques: Squeezing the
     * Silicon", introduction: the FP16/quantization pillar; ninfer pull
     * request #160: narrow weight codes streamed through a TMA ring). Layers
     * 2..L multiply OCP E4M3 weights with E4M3 activations on the tensor
     * cores (FP32 accumulation): the weights are rounded once at pack time,
     * each hidden layer's FP16 activation is rounded to E4M3 (nearest even,
     * saturating at +-448) as it is stored for the next layer. Layer 1, the
     * biases and every layer's FP16 result and activation are as in the other
     * variants. The weights always stream through the shared ring.
     * Available when L >= 2 and every hidden width (dims[1] .. dims[L-1]) is
     * a multiple of 32; otherwise nm_mlp_set_variant and nm_mlp_plan return
     * NM_ERR_UNSUPPORTED. */
    NM_VARIANT_FP8_WEIGHTS = 4
} nm_variant;

/* Version of this ABI (bumped on any incompatible change). */
int32_t nm_abi_version(void);

/* Human-readable name of a status code (static string, never NULL). */
const char *nm_status_str(nm_status s);

/* Create a network of L = n_dims - 1 affine layers with widths
 * dims[0] (inputs) .. dims[L] (outputs).
 * Supported: 1 <= L <= 16 and every width a multiple of 16 in [16, 256].
 * Allocates the packed blob and a status word on the current device (the
 * handle owns them; nm_mlp_destroy frees them).
 * Errors: NM_ERR_INVALID_ARG (dims or out NULL, n_dims < 2),
 * NM_ERR_UNSUPPORTED (widths/depth outside the set above, or the current
 * device is not compute capability 10.3), NM_ERR_OOM, NM_ERR_CUDA.
 * On error *out is set to NULL. */
nm_status nm_mlp_create(const int32_t *dims, int32_t n_dims, nm_mlp **out);

/* Size in bytes of the packed (device-private) weight blob -- the analogue of
 * the page's size query for the InferencingOptimal layout. */
nm_status nm_mlp_packed_size(const nm_mlp *h, size_t *bytes);

/* One-time conversion of the canonical weights into the packed layout
 * ("Row-major versus InferencingOptimal weights").
 * W: host array of L device pointers; W[l] is FP16 [dims[l+1]][dims[l]]
 *    row-major (row o holds the weights of output o).
 * b: host array of L device pointers; b[l] is FP16 [dims[l+1]].
 * The packed bits are a permutation of the input bits (no arithmetic). When
 * the handle's variant is NM_VARIANT_FP8_WEIGHTS the call also writes the
 * E4M3 images (nm_mlp_packed_fp8), rounding every weight of W_2 .. W_L to
 * E4M3; otherwise the first dispatch of that variant writes them, from the
 * packed blob, on its own stream (that first dispatch cannot be captured
 * into a CUDA graph: see nm_mlp_infer).
 * Errors: NM_ERR_INVALID_ARG (NULL or misaligned pointer), NM_ERR_CUDA. */
nm_status nm_mlp_pack_weights(nm_mlp *h, const void *const *W, const void *const *b,
                              nm_stream stream);

/* The E4M3 weight images of NM_VARIANT_FP8_WEIGHTS, kept beside the packed
 * blob (same allocation, owned by the handle): device address and size in
 * bytes (read-only; for byte-for-byte checks).
 * Layout: the images of W_2 .. W_L in order, each starting at a multiple of
 * 1024 bytes; an image's k range is cut into 128-, then 64-, then 32-column
 * segments (1024-aligned, N rows of w bytes, 128/64/32-byte swizzle).
 * Errors: NM_ERR_INVALID_ARG, NM_ERR_UNSUPPORTED (the network has no such
 * images: L < 2 or a hidden width not a multiple of 32), NM_ERR_NOT_PACKED
 * (not written since the last pack: see nm_mlp_pack_weights). */
nm_status nm_mlp_packed_fp8(const nm_mlp *h, const void **region, size_t *bytes);

/* Inverse of nm_mlp_pack_weights, into caller buffers of the same shapes.
 * Errors: NM_ERR_INVALID_ARG, NM_ERR_NOT_PACKED, NM_ERR_CUDA. */
nm_status nm_mlp_unpack_weights(const nm_mlp *h, void *const *W, void *const *b,
                                nm_stream stream);

/* Device address of the packed blob (read-only; for byte-for-byte checks of
 * the packer). Valid until nm_mlp_destroy. */
nm_status nm_mlp_packed_blob(const nm_mlp *h, const void **blob);

/* Evaluate the network on n inputs ("Experiment setup": one dispatch).
 * in:  device FP16 [n][dims[0]] row-major.   out: device FP16 [n][dims[L]].
 * n == 0 is a no-op. Rows of `out` beyond n are never written.
 * Errors: NM_ERR_INVALID_ARG (NULL/misaligned pointers, n < 0 or n > 2^31 - 128),
 * NM_ERR_NOT_PACKED, NM_ERR_UNSUPPORTED (the network does not fit the
 * selected variant's shared-memory budget), NM_ERR_CUDA (launch failure).
 * A kernel-side wait that gives up is reported by nm_mlp_device_status.
 * The first dispatch of the row-major variant, and of the narrow-precision
 * variant after a pack made with another variant selected, first converts
 * the weights once (a row-major copy, or the E4M3 images); it returns
 * NM_ERR_UNSUPPORTED, before enqueuing anything, if `stream` is being
 * captured into a CUDA graph (make one such dispatch before capturing).
 * Stream order: the dispatch is launched with programmatic stream
 * serialisation. Its set-up (barriers, tensor memory, weight staging) may
 * run while the previous kernel on `stream` finishes. It reads `in` and
 * writes `out` only after that kernel has completed, so chaining dispatches
 * through shared buffers on one stream is safe. A dispatch that directly
 * follows this handle's nm_mlp_pack_weights on the same stream does not
 * overlap it. */
nm_status nm_mlp_infer(nm_mlp *h, const void *in, int64_t n, void *out, nm_stream stream);

/* The same evaluation with the inputs and outputs in HOST memory. The pages
 * have no counterpart (their dispatch reads a batch already on the device);
 * it serves callers whose samples live on the host, so that the copies in
 * and out overlap the kernel instead of preceding and following it.
 * host_in:  FP16 [n][dims[0]] row-major.  host_out: FP16 [n][dims[L]].
 * Page-locked host memory (cudaHostAlloc / cudaHostRegister) lets the copies
 * run asynchronously; pageable memory works but serialises them.
 * The rows are processed in chunks (a multiple of 128 rows, see
 * nm_mlp_set_host_chunk) on three streams the handle owns: chunk i's
 * host-to-device copy, kernel and device-to-host copy run in order on
 * stream i % 3, so the copies of neighbouring chunks overlap its kernel.
 * Staging buffers for three chunks are allocated on the first call and kept
 * by the handle. The work is ordered after everything already enqueued on
 * `stream`, and `stream` waits for all of it: the host buffers must stay
 * valid, and host_out must not be read, until `stream` reaches that point.
 * Calls on one handle are serialised on its streams (safe, not concurrent).
 * The results are bit-identical to nm_mlp_infer on the same rows.
 * Errors: NM_ERR_INVALID_ARG (NULL pointer, n < 0 or n > 2^31 - 128),
 * NM_ERR_NOT_PACKED, NM_ERR_UNSUPPORTED, NM_ERR_OOM (staging buffers),
 * NM_ERR_CUDA. A kernel-side give-up is reported by nm_mlp_device_status. */
nm_status nm_mlp_infer_host(nm_mlp *h, const void *host_in, int64_t n, void *host_out,
                            nm_stream stream);

/* Rows per chunk of nm_mlp_infer_host: a multiple of 128 in [128, 2^20], or
 * 0 for the default (about 12 MiB of input per chunk, at least 16,384 rows).
 * Changing it frees the staging buffers (after the handle's streams drain);
 * the next call allocates them anew. Errors: NM_ERR_INVALID_ARG. */
nm_status nm_mlp_set_host_chunk(nm_mlp *h, int64_t rows);

/* Select the kernel variant used by later nm_mlp_infer calls.
 * Errors: NM_ERR_INVALID_ARG for an unknown variant, NM_ERR_UNSUPPORTED for
 * NM_VARIANT_FP8_WEIGHTS on a network without E4M3 images. */
nm_status nm_mlp_set_variant(nm_mlp *h, nm_variant v);

/* Synchronise `stream`, then read and clear the handle's device status word.
 * Returns NM_ERR_RANGE_CHECK if (checking build) a kernel of this handle
 * found an address outside its plan's tensor or shared memory,
 * NM_ERR_TIMEOUT if one gave up a bounded wait since the last call (its
 * outputs are then undefined), NM_ERR_CUDA if the synchronisation reported an
 * error, else NM_OK. */
nm_status nm_mlp_device_status(nm_mlp *h, nm_stream stream);

/* Limit, in nanoseconds, of every wait inside the inference kernels
 * (default 2,000,000,000). A wait that exceeds it sets the status word and
 * the kernel winds down (drains its copies in flight, frees its tensor
 * memory) and returns. Tests set a tiny limit to exercise that path. */
nm_status nm_mlp_set_wait_limit(nm_mlp *h, uint64_t nanoseconds);

/* Test hook for the failure path. With `enable` non-zero, every CTA of later
 * nm_mlp_infer launches first waits on a barrier that nothing ever signals,
 * so that wait runs out after the wait limit: the kernel then takes its
 * give-up path (status word set, copies drained, tensor memory freed) without
 * any fault. The outputs of such a launch are undefined. */
nm_status nm_mlp_set_test_stall(nm_mlp *h, int32_t enable);

/* The checking build. The library can be compiled with NM_RANGE_CHECKS
 * defined (libnmmlp_check.so; `python -m mlp_neural_gb300.build --checked`):
 * its kernels then compare every tensor-memory column range they load,
 * store or accumulate into (against the columns the plan uses), and every
 * shared-memory range a copy or store writes (against the end of the plan's
 * shared-memory layout, and each copy against its buffer), and record a
 * miss in the status word, reported by nm_mlp_device_status as
 * NM_ERR_RANGE_CHECK, without changing what they access: a stand-in for a
 * memory checker over the memories such a tool does not see.
 * nm_checking_build returns 1 in that build, 0 otherwise. */
int32_t nm_checking_build(void);

/* Test hook of the checking build: compare tensor-memory columns with
 * `tmem_columns` instead of the plan's (0 restores the plan's; a limit above
 * the plan's is ignored), so that a test can see a check fire without any
 * access changing. No effect in the normal build. Errors:
 * NM_ERR_INVALID_ARG (null handle). */
nm_status nm_mlp_set_test_check_limit(nm_mlp *h, uint32_t tmem_columns);

/* Inference that allocates no device memory. The source pages have no
 * counterpart to this call; it exists for callers that cannot call
 * cudaMalloc -- code embedded in a host application that owns the device's
 * whole memory budget, or a latency-critical path where an allocation's
 * implicit synchronisation is not allowed -- but that can pass device buffers
 * they already own.
 * W, b: host arrays of L device pointers to the row-major FP16 weights
 *       [dims[l+1]][dims[l]] and biases [dims[l+1]] (as for pack_weights);
 * in, out, n, stream: as for nm_mlp_infer.
 * Every call packs the weights again and runs the fused kernel (fused
 * variant) out of one library-owned, file-scope device array of 1 MiB, which
 * every GPU that loads the library holds until the process exits. Networks
 * whose packed weights and biases exceed 1,043,456 bytes are rejected with
 * NM_ERR_UNSUPPORTED (the page-shaped network needs 58,272; the widest
 * 256-wide 16-layer network would need about 2 MB).
 * The first call on a device looks up that array's device address with the
 * device current (a one-time set-up). All calls share the array and it keeps
 * the last call's contents (each call clears what must start at zero): calls
 * whose work overlaps on the GPU -- from several host threads, or on several
 * streams -- race and must not be made.
 * The call returns after `stream` has completed the work (it synchronises the
 * stream), so a kernel-side give-up is reported directly as NM_ERR_TIMEOUT
 * (and, in the checking build, a failed range check as NM_ERR_RANGE_CHECK).
 * Because it synchronises, it refuses a stream that is being captured into a
 * CUDA graph: it then returns NM_ERR_UNSUPPORTED before enqueuing anything.
 * Errors: NM_ERR_INVALID_ARG, NM_ERR_UNSUPPORTED, NM_ERR_CUDA, NM_ERR_TIMEOUT,
 * NM_ERR_RANGE_CHECK (checking build only). */
nm_status nm_mlp_infer_noalloc(const int32_t *dims, int32_t n_dims, const void *const *W,
                               const void *const *b, const void *in, int64_t n, void *out,
                               nm_stream stream);

/* How the fused kernel runs a network, worked out on the host alone: no
 * device is touched, so this answers on a machine without a GPU. The kernel
 * keeps several 128-sample tiles in flight per CTA (tile slots), as many as
 * tensor memory allows; it keeps the packed weights resident in shared
 * memory when they fit, and otherwise streams them through a shared ring.
 * nm_mlp_infer uses the same plan for the same widths, variant and shared
 * memory limit.
 * dims, n_dims: as for nm_mlp_create.
 * variant: the kernel variant (nm_mlp_set_variant).
 * smem_optin: the device's opt-in shared memory per block, in bytes
 *   (cudaDevAttrMaxSharedMemoryPerBlockOptin; 232,448 on GB300).
 * The row-major ablation never stages the packed weights: it rebuilds each
 * layer's operand per tile, so its plans report streamed_weights = 0.
 * Errors: NM_ERR_INVALID_ARG (NULL pointer, fewer than two widths, unknown
 * variant), NM_ERR_UNSUPPORTED (a width or layer count out of range, or no
 * plan fits in smem_optin; nm_mlp_infer then answers the same). */
typedef struct nm_plan {
  int32_t tile_slots;       /* 128-sample tiles in flight per CTA */
  int32_t warps_per_slot;   /* epilogue warps: 4 TMEM lane quadrants x column groups */
  int32_t threads;          /* per CTA. Resident weights: 8 warps (one issuing warp per
                               slot, the input producer, the rest idle) plus the slots'
                               epilogue warps. Streamed weights: the slots' warps (which
                               also issue), the weight producer and the input producer. */
  int32_t streamed_weights; /* 0: resident in shared memory, 1: streamed */
  int32_t weight_stages;    /* depth of the streamed-weight ring (0 if resident) */
  int32_t input_stages;     /* input ring stages per slot */
  int32_t output_buffers;   /* output staging buffers per slot */
  uint32_t smem_bytes;      /* dynamic shared memory per CTA */
  uint32_t tmem_columns;    /* tensor memory columns allocated per CTA */
  int32_t issuing_warps;    /* warps that issue MMA chains (one per slot, or per pair of
                               slots with NM_VARIANT_PAIRED_TILES) */
  int32_t a_tmem_k;         /* columns of the next layer's A kept in tensor memory; a
                               streamed FP16 plan may keep the rest (whole 64-column
                               segments) in shared memory to fit one more tile slot */
} nm_plan;

nm_status nm_mlp_plan(const int32_t *dims, int32_t n_dims, nm_variant variant,
                      uint32_t smem_optin, nm_plan *plan);

/* Free the handle and its device memory (synchronises the device first).
 * NULL is a no-op. */
void nm_mlp_destroy(nm_mlp *h);

#ifdef __cplusplus
}
#endif

#endif /* NM_MLP_H */
