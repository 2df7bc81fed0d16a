/*
 * echo.h -- C ABI of libecho.so: the Echo error-compensated low-bit all-reduce,
 * with P tensor-parallel ranks emulated as P buffers in one GPU's memory.
 *
 * The operation is the quantized P2P all-reduce of "Echo: Error-Compensated
 * 4-Bit Tensor-Parallel Communication for LLM Training and Inference" (arXiv
 * 2610.14277), Fig. 2(a), with the error feedback described in its abstract and
 * in the article "Your All-Reduce Is 4x Overpriced: Echo's 4-Bit Error-Feedback
 * Trick for Tensor-Parallel Training" (section "The cancellation rule"):
 *
 *   push    every rank p quantizes each segment it does not own (after adding
 *           the error it holds for those elements) to b-bit codes with one fp16
 *           step and one fp16 zero point per group of g elements, and writes
 *           them to that segment owner's receive slot;
 *   reduce  the owner of segment o decodes the P-1 received code tiles and sums
 *           them with its own segment (plus its held error) in fp32, in
 *           ascending rank order;
 *   gather  the owner quantizes the sum once; every rank, the owner included,
 *           decodes the same codes, so all P outputs are bit-identical and every
 *           element passes through at most two quantizers for any P;
 *   feedback each error the call reveals is kept where it arose (the sender's
 *           stage-1 error v - deq(q) on its non-owned elements, the owner's
 *           stage-2 error sum - output on its own segment) and is added back by
 *           the next call's entry pass.
 *
 * The quantizer (zero-aware asymmetric, the paper's Table 8 "full" row; its
 * formula is not printed on the pages) is read as: lo = min(0, min v),
 * hi = max(0, max v), s = fp16 round-up of (hi - lo) / (2^b - 1) (1 for an
 * all-zero group), z = clamp(rint(-lo / s), 0, 2^b - 1),
 * q = clamp(rint(v / s) + z, 0, 2^b - 1), decoded as s * (q - z); all in IEEE
 * fp32 with no fused multiply-add.  Outputs are rounded to bf16 (nearest even).
 *
 * ---------------------------------------------------------------------------
 * Conventions for every call
 *   - Device pointers are plain CUDA device addresses on the device that was
 *     current when the plan was made; that device must be current at each call.
 *   - `stream` is a cudaStream_t passed as void* (NULL = the legacy default
 *     stream).  Work is enqueued on it and the call returns without waiting,
 *     except where a call says it synchronizes.
 *   - Every call returns an ECHO_* status; 0 is success.  On ECHO_ERR_CUDA the
 *     CUDA error is kept and echo_strerror(ECHO_ERR_CUDA) names it.
 *   - A plan serves one stream at a time: its receive slots are shared by all
 *     calls made with it, so calls on different streams must be ordered by the
 *     caller.  Distinct plans are independent.
 * ---------------------------------------------------------------------------
 */
#ifndef ECHO_H_
#define ECHO_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Status codes. */
#define ECHO_OK              0
#define ECHO_ERR_ARG         1  /* NULL pointer, P outside 1..ECHO_MAX_RANKS, g < 1,
                                   aliasing other than out[p] == in[p], wrong device */
#define ECHO_ERR_SHAPE       2  /* n < 0, or n not a multiple of P*g */
#define ECHO_ERR_UNSUPPORTED 3  /* bits not 4 or 8, or g not 64, 128 or 256 */
#define ECHO_ERR_ALIGN       4  /* an input or output not 16-byte aligned, or a
                                   compensator state not 32-byte aligned */
#define ECHO_ERR_CUDA        5  /* a CUDA runtime call failed */
#define ECHO_ERR_OVERFLOW    6  /* (status word) a non-finite input or an fp16 step overflow */
#define ECHO_ERR_TIMEOUT     7  /* (status word) a device-side wait gave up */
#define ECHO_ERR_TOO_LARGE   8  /* echo_allreduce_noalloc: beyond its fixed scratch area */

#define ECHO_MAX_RANKS 16

/* Pass as `comp_state` to use the compensator state owned by the plan. */
#define ECHO_COMP_DEFAULT ((void*)(intptr_t)-1)

typedef struct echo_plan_s* echo_plan_t;

/*
 * echo_plan -- build the layout for P emulated ranks of n bf16 elements each,
 * groups of g elements and b-bit codes, and allocate (cudaMalloc, on the
 * current device) the plan's receive slots and its own compensator state
 * (P*n fp32, zeroed; room enough for either format of echo_set_state).  Synchronizes the device once.
 *   P     1..ECHO_MAX_RANKS
 *   n     elements per rank, a multiple of P*g (n = 0 gives an empty plan)
 *   g     elements per group: 128 (the method's), or 64 or 256 (the group-size
 *         rows of the paper's Table 8 ablation); wire codes take g*b/8 bytes
 *         and one 4-byte meta word per group
 *   bits  4 or 8
 *   out   receives the plan handle; the caller frees it with echo_plan_destroy.
 * Segments are contiguous: rank o owns elements [o*m, (o+1)*m), m = n/P
 * (Fig. 2(a) and Fig. 4 of the paper show contiguous segments).
 */
int echo_plan(int P, int64_t n, int g, int bits, echo_plan_t* out);

/*
 * echo_allreduce -- one emulated all-reduce call (Fig. 2(a)).
 *   in[P]       host array of P device pointers, each to n bf16 values (rank p's
 *               partial tensor), 16-byte aligned, caller-owned, read-only.
 *   out[P]      host array of P device pointers, each to n bf16 outputs, 16-byte
 *               aligned, caller-owned.  All P rows receive the same bits.
 *               out[p] may equal in[p] (in place); any other overlap between an
 *               out buffer and another in/out buffer is rejected (ECHO_ERR_ARG).
 *   comp_state  NULL: uncompensated call (no state read or written);
 *               ECHO_COMP_DEFAULT: the plan's own state;
 *               otherwise a caller device buffer of echo_comp_bytes(plan) bytes,
 *               32-byte aligned, laid out [P][n] (rank p's error for its
 *               element i at p*n + i) in fp32, or bf16 or fp16 after
 *               echo_set_state,
 *               zero before the first call of a sequence;
 *               read and updated in place.
 *   stream      cudaStream_t as void*.
 * Enqueues one kernel (a block per owner tile, see echo_set_tile_fused; two,
 * push then reduce, with echo_set_tile_fused 0; three with a separate gather
 * kernel, see echo_set_fused; one persistent kernel with echo_set_persistent)
 * and returns.  Inputs must stay valid and
 * unmodified until the work completes.  Non-finite inputs or an fp16 step
 * overflow do not fail the call: they set the plan's status word (see
 * echo_get_status) and leave the affected groups' results unspecified.
 */
int echo_allreduce(echo_plan_t plan, const void* const* in, void* const* out,
                   void* comp_state, void* stream);

/*
 * echo_reset_comp -- zero the plan's own compensator state, ordered on the
 * stream of the plan's last echo_allreduce (the legacy default stream if none).
 */
int echo_reset_comp(echo_plan_t plan);

/*
 * echo_reset_comp_async -- zero a compensator state on `stream`.
 * comp_state is ECHO_COMP_DEFAULT or a caller buffer of echo_comp_bytes bytes.
 */
int echo_reset_comp_async(echo_plan_t plan, void* comp_state, void* stream);

/* Bytes of one compensator state: P * n * 4 (fp32 state, the default) or
 * P * n * 2 (bf16 or fp16 state, see echo_set_state).  0 for a NULL plan. */
size_t echo_comp_bytes(echo_plan_t plan);

/* Bytes of the plan's receive-slot workspace (what echo_debug_wire copies). */
size_t echo_wire_bytes(echo_plan_t plan);

/*
 * echo_wire_layout -- describe the receive-slot workspace, for tests and tools.
 * Writes 8 int64 values to `desc`:
 *   [0] byte offset of the push codes    [P owners][P-1 senders][Gs groups][g*b/8 bytes]
 *   [1] byte offset of the push meta     [P owners][P-1 senders][Gs_pad] uint32
 *   [2] byte offset of the gather codes  [P owners][Gs groups][g*b/8 bytes]
 *   [3] byte offset of the gather meta   [P owners][Gs_pad] uint32
 *   [4] Gs     groups per segment (m / g)
 *   [5] Gs_pad Gs rounded up to a multiple of 4
 *   [6] bytes of codes per group (g * b / 8)
 *   [7] total bytes (echo_wire_bytes)
 * Sender slot index: rank p's slot at owner o is p if p < o, else p - 1.
 * A meta word holds the fp16 step in its low 16 bits and the fp16 zero point
 * (an integer value) in its high 16 bits.  Codes of 4 bits: element 2i of a
 * group in the low nibble of byte i, element 2i+1 in the high nibble.
 */
int echo_wire_layout(echo_plan_t plan, int64_t* desc);

/*
 * echo_get_status -- read and clear the plan's device status word.
 * Synchronizes `stream`, then writes ECHO_OK, ECHO_ERR_OVERFLOW or
 * ECHO_ERR_TIMEOUT (the latter wins if both occurred) to *status.
 */
int echo_get_status(echo_plan_t plan, void* stream, int* status);

/*
 * echo_debug_wire -- copy the whole receive-slot workspace (layout as in
 * echo_wire_layout) to host memory `host_dst` of at least `bytes` bytes, after
 * the work already on `stream`.  Synchronizes `stream`.  For tests.
 */
int echo_debug_wire(echo_plan_t plan, void* host_dst, size_t bytes, void* stream);

/*
 * echo_set_fused -- 1 (default): the block that encodes the gather codes
 * (the tile-fused kernel's, or the reduce kernel's) writes the P outputs
 * itself from the values it has just encoded (the gather codes are still
 * written); with every rank's output in this GPU's memory, that is the
 * all-gather's decode without a second read of the codes or another kernel.
 * 0: push, reduce and a separate gather kernel, which reads the gather codes
 * back and writes all P outputs, as each receiving rank would.  All give
 * bit-identical outputs, state and codes.
 */
int echo_set_fused(echo_plan_t plan, int fused);

/*
 * echo_set_timing -- events (cudaEvent_t as void*) that echo_allreduce records
 * around its kernels: ev[0] before the push kernel, ev[1] after it, ev[2] after
 * the reduce kernel, ev[3] after the gather kernel (== after reduce when
 * fused); with one kernel per call (tile-fused or persistent) ev[1..3] are
 * all recorded after it.  count 4 enables, count 0 disables.  The caller owns
 * the events.
 */
int echo_set_timing(echo_plan_t plan, void* const* events, int count);

/*
 * echo_allreduce_noalloc -- the same call as echo_allreduce, for callers that
 * must not allocate device memory.  The paper has no counterpart: this is an
 * interface of this library only.
 *
 * Who needs it: code that runs where another component owns the device memory
 * budget and forbids allocation on the execution path (a plugin inside an
 * inference runtime, for one), and latency-critical loops where cudaMalloc's
 * implicit device synchronization, or an allocation failing late on a nearly
 * full device, is not acceptable.  echo_plan allocates its receive slots and
 * state with cudaMalloc; this entry point needs no plan and allocates nothing.
 *
 * Scratch: the receive slots live in one file-scope __device__ array of
 * ECHO_NOALLOC_SCRATCH_BYTES (32 MiB).  Every GPU that loads the library's
 * device code holds it until the process exits (with CUDA's default lazy
 * module loading, from this entry point's first call on that GPU).  The first call on a device looks the array's
 * device address up (cudaGetSymbolAddress) and sets the kernels' attributes,
 * with that device current; make that first call before any stream capture.
 * Every call on a device shares the array and leaves the last call's codes in
 * it (the call clears what must start at zero itself), so calls whose work
 * overlaps on the GPU -- on different streams, or from different threads
 * without ordering -- race.  Calls on one stream are ordered and safe.
 *
 *   P, n, bits  as for echo_plan, with g = 128.  A problem whose receive slots
 *               (about P*n*(b/8 + 4/128) bytes, see echo_wire_layout) do not
 *               fit the array returns ECHO_ERR_TOO_LARGE; for example P=4 with
 *               4-bit codes fits up to 2048 x 4096 elements per rank.
 *   in, out     as for echo_allreduce (same alignment and aliasing rules).
 *   comp_state  NULL (uncompensated) or a caller device buffer of P*n*4 bytes,
 *               32-byte aligned,
 *               fp32 [P][n], as for echo_allreduce; ECHO_COMP_DEFAULT is
 *               rejected (ECHO_ERR_ARG) since there is no plan.
 *   stream      cudaStream_t as void*.
 * Two kernels (push, then reduce writing the outputs).  Outputs, state and
 * codes are bit-identical to echo_allreduce's.  Non-finite inputs are not
 * reported: there is no status word to read back.
 */
#define ECHO_NOALLOC_SCRATCH_BYTES ((size_t)32 << 20)
int echo_allreduce_noalloc(int P, int64_t n, int bits, const void* const* in,
                           void* const* out, void* comp_state, void* stream);

/*
 * echo_set_tile_fused -- ECHO_TILE_AUTO (1, the default): run each
 * echo_allreduce of the plan as one kernel in which a block computes a whole
 * owner tile; ECHO_TILE_OFF (0): as two kernels, the push, then the reduce
 * (which also writes the outputs).  The push of the P-1 senders, the owner's
 * sum and the gather of a tile of a segment (Fig. 2(a)) read and write only
 * that tile's element positions of
 * the P ranks, so with every rank in one GPU's memory one block can take all
 * of them, with no block waiting on another and no kernel boundary between
 * the push and the reduce.  The block walks the ranks in ascending order:
 * each sender's codes and meta word are written to the owner's receive slot
 * and its held error updated, as by the push; the owner sums the decoded
 * values (decoding the codes it has just encoded rather than reading the slot
 * back) with its own segment in fp32, quantizes the sum once, writes the
 * gather codes and every rank's output and keeps its error.  Results, state
 * and receive slots are bit-identical to the other schedules.  It applies
 * while the gather is fused (echo_set_fused 1, the default) and the call is
 * not persistent (echo_set_persistent 0, the default): a separate gather
 * kernel or the persistent kernel take precedence.
 * The kernel has two forms with the same results.  In the rank loop a small
 * block walks the ranks one after another, many blocks per SM; in the
 * rank-parallel form a block has a warp pair per rank, which push their
 * ranks at the same time, and the sum and gather follow, so a block's path is
 * one push long instead of P.  ECHO_TILE_AUTO takes the rank-parallel form
 * when the call's blocks (one per 1024 elements of a rank) are at most four
 * times the device's SMs and P >= 2, the rank loop otherwise;
 * ECHO_TILE_RANK_LOOP (2) and ECHO_TILE_RANK_PARALLEL (3) force one form (the
 * rank-parallel form for P up to 16).  ECHO_ERR_ARG for other values of on.
 */
#define ECHO_TILE_OFF           0
#define ECHO_TILE_AUTO          1
#define ECHO_TILE_RANK_LOOP     2
#define ECHO_TILE_RANK_PARALLEL 3
int echo_set_tile_fused(echo_plan_t plan, int on);

/*
 * echo_set_persistent -- run each later echo_allreduce of the plan as one
 * persistent kernel instead of two or three kernels (on = 1), or back
 * (on = 0).
 * The paper overlaps the push, reduce and gather of different tiles
 * (Fig. 2(b)); here every (sender, owner, tile) push, every reduce tile and
 * every gather tile is a work item that blocks claim in order from an atomic
 * ticket counter, and a reduce tile starts as soon as its P-1 pushes are done
 * (a gather tile as soon as its reduce is), with per-tile counters in the
 * plan.  Results are bit-identical to the three-kernel path, with or without
 * the fused gather.  The launch is cooperative (every block resident).  Every
 * device-side wait is bounded (1 s); a call that gives up sets the status word
 * to ECHO_ERR_TIMEOUT and leaves its results unspecified, and the following
 * echo_get_status clears the plan's schedule words so that the next call
 * starts clean.  Returns ECHO_ERR_UNSUPPORTED for a problem with 2^31 or more
 * work items, ECHO_ERR_ARG for on not 0 or 1.
 */
int echo_set_persistent(echo_plan_t plan, int on);

/*
 * echo_debug_hold_push -- test hook for the bounded waits of the persistent
 * kernel: in every later persistent call, the push work item with ticket
 * `item` (0-based; items are ordered tile by tile, then by sender and owner)
 * does its work but never reports it, so the reduce of its tile waits until
 * its bound and the call ends with ECHO_ERR_TIMEOUT.  -1 (the default) turns
 * the hook off.  ECHO_ERR_ARG for item < -1.
 */
int echo_debug_hold_push(echo_plan_t plan, int64_t item);

/*
 * echo_set_quantizer -- choose the group quantizer of a plan's calls.
 *   ECHO_QUANT_ZERO_AWARE (default): the method's zero-aware asymmetric
 *     quantizer (the "full" row of the paper's Table 8), as described at the
 *     top of this header.
 *   ECHO_QUANT_NAIVE_ZERO_POINT, ECHO_QUANT_SYMMETRIC: the two ablation rows of
 *     Table 8 ("naive zero-point", "symmetric grid"), whose formulas are not
 *     printed either; read as
 *       naive:     range [min v, max v] without 0, an fp16 offset m rounded
 *                  down from min v (carried in the meta word's zero-point
 *                  half), s = (max v - m)/(2^b - 1) rounded up to fp16,
 *                  q = clamp(rint((v - m)/s), 0, 2^b - 1), decoded m + s*q;
 *       symmetric: s = max|v|/(2^(b-1) - 1) rounded up to fp16, zero point
 *                  2^(b-1), q = clamp(rint(v/s), +-(2^(b-1) - 1)) + 2^(b-1).
 * Applies to both quantizations of every later echo_allreduce of the plan;
 * the wire layout is unchanged.  Any other value returns ECHO_ERR_ARG.
 */
#define ECHO_QUANT_ZERO_AWARE       0
#define ECHO_QUANT_NAIVE_ZERO_POINT 1
#define ECHO_QUANT_SYMMETRIC        2
int echo_set_quantizer(echo_plan_t plan, int mode);

/*
 * echo_set_state -- choose how a plan's calls keep the compensator state (the
 * reduced-precision and decayed variants of the error feedback; the article's
 * section "The cancellation rule" names a two-timescale compensator but no
 * page prints its equations, its precision or a decay constant, so both
 * options are readings):
 *   format  ECHO_STATE_F32 (default): each kept error is an fp32 value;
 *           ECHO_STATE_BF16: each kept error is rounded to bf16 (nearest
 *           even) when stored, halving the state's size and traffic;
 *           ECHO_STATE_F16: the same with fp16 (nearest even): 3 more
 *           significand bits than bf16 but a range that ends at 65504 and
 *           turns subnormal below 6.1e-5, where small errors lose precision.
 *   decay   the kept error is fl32(decay * r) for each revealed error r (then
 *           rounded to bf16 under ECHO_STATE_BF16); 1 (default) is plain
 *           error feedback, below 1 a leaky one.  Must be finite, in (0, 1].
 * The state layout stays [P][n] (element i of rank p at p*n + i) in the chosen
 * type; echo_comp_bytes(plan) becomes P*n*4 or P*n*2 accordingly, and a caller
 * state passed to echo_allreduce must hold that many bytes in that type.
 * Changing the format zeroes the plan's own state (ordered as
 * echo_reset_comp); changing only the decay keeps it.  Invalid values return
 * ECHO_ERR_ARG and leave the plan unchanged.
 */
#define ECHO_STATE_F32  0
#define ECHO_STATE_BF16 1
#define ECHO_STATE_F16  2
int echo_set_state(echo_plan_t plan, int format, float decay);

/*
 * echo_debug_set_grid -- debug: launch every kernel of the plan's later calls
 * with at most `blocks` blocks along the dimension its blocks stride over
 * (0, the default: the launchers' own choice).  The kernels stride, so any
 * grid computes the same bits; tests compare a 1-block grid with the default
 * one to catch indexing that depends on the grid.  ECHO_ERR_ARG for blocks < 0.
 */
int echo_debug_set_grid(echo_plan_t plan, int blocks);

/*
 * echo_debug_check_guards -- debug: the plan's receive slots and its own
 * compensator state are allocated with a 256-byte guard band on each side,
 * filled with a fixed byte at plan time.  Writes 1 to *intact if all four
 * bands still hold it (no kernel wrote outside its buffers), else 0.
 * Synchronizes the device.
 */
int echo_debug_check_guards(echo_plan_t plan, int* intact);

/* Free everything the plan allocated.  NULL is accepted. */
void echo_plan_destroy(echo_plan_t plan);

/* A static description of a status code; for ECHO_ERR_CUDA, of the last CUDA
 * error seen by the library in this thread. */
const char* echo_strerror(int status);

#ifdef __cplusplus
}
#endif

#endif /* ECHO_H_ */
