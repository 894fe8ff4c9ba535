/*
 * lst.h - layer-streamed optimizer update over packed per-layer state blocks.
 *
 * C ABI of liblst.so (GB300, sm_103a). Plain pointers and sizes only.
 *
 * The method. Training state (weights W, gradients G, Adam moments m, v and,
 * in one layout, an fp32 master copy of W) lives in one contiguous block per
 * transformer layer. The optimizer updates each block with the per-parameter
 * Adam rule written as an additive delta on the stored weight
 *   m' = b1*m + (1-b1)*g,  v' = b2*v + (1-b2)*g^2,
 *   m^ = m'/(1-b1^t),      v^ = v'/(1-b2^t),
 *   W += -(lr * m^/(sqrt(v^) + eps))           (t: one global step counter)
 * ("Training 70B Models on Consumer Hardware (If You're Willing to Wait)",
 * section "The Math"), or with the SGD form W += (-lr*g) (same page, section
 * "The Assumption Everyone Makes"). Blocks are either resident in device
 * memory, or held in pinned host memory and streamed through the device one
 * layer at a time over two device buffers and three CUDA streams ordered by
 * events ("MegaTrain" summary page, sections on layer-contiguous memory
 * tiling, the double-buffered pipeline and three-stream execution).
 *
 * Arithmetic (both the device-resident and the streamed path compute exactly
 * this, so their results are bit-identical):
 *   - every step below is one IEEE fp32 operation, rounded to nearest, in this
 *     order, with no fused multiply-add:
 *       m = b1*m + omb1*g;  v = b2*v + omb2*(g*g);
 *       mh = m/bc1;  vh = v/bc2;  u = mh/(sqrt(vh) + eps);
 *       w = w*decay - lr*u
 *   - omb1 = 1-b1, omb2 = 1-b2, bc1 = 1-b1^t, bc2 = 1-b2^t and
 *     decay = 1 - lr*weight_decay are formed in double on the host and rounded
 *     once to fp32. Weight decay is decoupled (AdamW) and applied to the weight
 *     before the Adam step; the pages themselves give plain Adam.
 *   - bf16 values are widened exactly; bf16 results are the fp32 result
 *     rounded to nearest, ties to even.
 *   - SGD: w = w + (-(lr*g)); m and v are not touched, no decay.
 *
 * Layouts (per parameter; a block is segment-of-arrays, one segment per field,
 * in the order listed, each segment starting on a 4 KB boundary):
 *   LST_L12_BF16   G bf16 | W bf16 | m f32 | v f32                 12 B
 *   LST_L16_MIXED  G bf16 | master f32 | m f32 | v f32 | W bf16    16 B
 *                  (W is an output: the new master rounded to bf16)
 *   LST_L16_FP32   G f32 | W f32 | m f32 | v f32                   16 B
 * Within a block, tensors follow in the order given to lst_layout_create, each
 * starting at an element index that is a multiple of 8; the block's element
 * count is rounded up to a multiple of 2048. Padding elements must hold zero:
 * the update maps a zero element (g = W = m = v = 0) to zero, and the kernels
 * update padding along with the tensors.
 * G comes first and the output fields last, so the bytes sent host -> device
 * (the fields the update reads) are one prefix of the block, and the bytes
 * sent back (the fields it writes) are one suffix.
 *
 * Ownership: the caller owns all host and device memory and keeps it valid
 * for the duration of a call (and, for the asynchronous lst_adamw_step /
 * lst_sgd_step, until the work on the given stream has finished). The layout
 * handle is owned by the library and freed with lst_layout_destroy. The step
 * calls allocate no device memory.
 *
 * Errors: every call returns an lst_status and never aborts or exits. On
 * LST_ERR_CUDA the CUDA error text is available from lst_last_error() (per
 * thread). A call that fails validation touches no memory.
 *
 * Threads: a layout may be used from several threads for lst_adamw_step /
 * lst_sgd_step. lst_stream_step serialises itself per layout.
 */
#ifndef LST_H
#define LST_H

#include <stdint.h>

#if defined(__GNUC__)
#define LST_API __attribute__((visibility("default")))
#else
#define LST_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

typedef enum lst_status {
  LST_OK = 0,
  LST_ERR_INVALID_ARG = 1, /* null pointer, bad size, hyperparameter outside its domain */
  LST_ERR_ALIGNMENT = 2,   /* pointer not aligned as the call requires */
  LST_ERR_NOT_PINNED = 3,  /* host block not page-locked (pinned) host memory */
  LST_ERR_CUDA = 4,        /* a CUDA runtime call failed; see lst_last_error() */
  LST_ERR_OOM = 5,         /* host allocation failed */
  LST_ERR_TIMEOUT = 6,     /* lst_stream_step's host-side deadline passed */
  LST_ERR_IO = 7           /* a block file could not be read, written or flushed */
} lst_status;

typedef enum lst_format {
  LST_L12_BF16 = 0,  /* 12 B/param: bf16 W, bf16 G, fp32 m, v */
  LST_L16_MIXED = 1, /* 16 B/param: 12 B + fp32 master, bf16 W derived */
  LST_L16_FP32 = 2   /* 16 B/param: fp32 W, G, m, v */
} lst_format;

typedef enum lst_field {
  LST_FIELD_G = 0,
  LST_FIELD_W = 1,
  LST_FIELD_M = 2,
  LST_FIELD_V = 3,
  LST_FIELD_MASTER = 4 /* LST_L16_MIXED only */
} lst_field;

typedef struct lst_layout lst_layout; /* opaque, owned by the library */
typedef struct lst_store lst_store;   /* opaque, owned by the library */

/* AdamW hyperparameters. step = t >= 1, the global step counter ("The Math":
   one scalar t for all layers, incremented each batch). 0 <= beta < 1;
   lr, eps, weight_decay finite. */
typedef struct lst_adamw_hparams {
  float lr, beta1, beta2, eps, weight_decay;
  int64_t step;
} lst_adamw_hparams;

/* ------------------------------------------------------------------------
 * Block geometry ("MegaTrain" summary page, layer-contiguous memory tiling:
 * one contiguous, 4 KB-aligned block per transformer layer). Host only.
 * ------------------------------------------------------------------------ */

/* Build a layout from n_tensors tensor shapes.
   ndim[i] in 0..4; dims holds 4 entries per tensor (dims[4*i + k], entries
   beyond ndim[i] ignored; a dimension of 0 gives an empty tensor).
   layer_of_tensor[i] is the block the tensor belongs to; blocks are numbered
   0..L-1 and each must hold at least one tensor. n_tensors == 0 gives a
   layout with no blocks. The arrays are read during the call only.
   Errors: LST_ERR_INVALID_ARG (null pointers with n_tensors > 0, ndim out of
   range, negative dims, a block index < 0 or a block without tensors, a
   block larger than 2^40 elements, unknown format), LST_ERR_OOM. */
LST_API lst_status lst_layout_create(int32_t n_tensors, const int32_t* ndim, const int64_t* dims,
                             const int32_t* layer_of_tensor, lst_format fmt, lst_layout** out);

/* Free a layout (null is ignored). Not concurrently with a call using it. */
LST_API void lst_layout_destroy(lst_layout* layout);

/* Number of blocks, total parameters (without padding), and the largest
   block's size in bytes. Any output pointer may be null. */
LST_API lst_status lst_layout_info(const lst_layout* layout, int64_t* n_layers, int64_t* n_params,
                           int64_t* max_block_bytes);

/* One block: its size in bytes, its parameter count (no padding) and its
   padded element count (the length of each segment in elements). Outputs may
   be null. LST_ERR_INVALID_ARG if layer is out of range. */
LST_API lst_status lst_layout_block(const lst_layout* layout, int64_t layer, int64_t* bytes, int64_t* params,
                            int64_t* padded_elems);

/* Byte offset and size of one field's segment within a block.
   LST_ERR_INVALID_ARG if the field does not exist in the layout's format. */
LST_API lst_status lst_layout_segment(const lst_layout* layout, int64_t layer, int32_t field,
                              int64_t* byte_offset, int64_t* bytes);

/* Byte offset, within its block, of a tensor's data in one field's segment
   (for building views of the block), and the tensor's block and element
   offset (either output may be null). */
LST_API lst_status lst_layout_tensor(const lst_layout* layout, int32_t tensor, int32_t field,
                             int64_t* byte_offset, int64_t* layer, int64_t* elem_offset);

/* The contiguous byte ranges of a block that the streamed step sends to the
   device (the fields the update reads) and copies back (the fields it
   writes). The gradient is never copied back. */
LST_API lst_status lst_layout_transfer(const lst_layout* layout, int64_t layer, int64_t* h2d_offset,
                               int64_t* h2d_bytes, int64_t* d2h_offset, int64_t* d2h_bytes);

/* Element count of the sub-chunks the streamed step moves and updates at a
   time (a multiple of 2048; 0 = one chunk per block). Default 16,777,216. */
LST_API lst_status lst_layout_set_stream_chunk(lst_layout* layout, int64_t elems);

/* How the streamed steps (lst_stream_step and its variants) move sub-chunks,
   per direction (the pages' StreamIn / StreamOut):
     LST_COPY_ENGINE  cudaMemcpyAsync / cudaMemcpy2DAsync on the copy engines;
     LST_COPY_SM      a copy kernel on the same stream that reads or writes the
                      host block through its device mapping (pinned memory
                      registered as mapped, e.g. from lst_host_alloc);
     LST_COPY_AUTO    the copy engines, except for the sub-chunks of a host
                      block that they moved slowly in an earlier streamed
                      step. Each step times every sub-chunk copy the copy
                      engines make (events on the copy streams); a sub-chunk
                      of 4 MB or more that took longer than 2.5x its bytes at
                      the best sub-chunk rate seen in its direction is moved
                      by the copy kernel in the later steps, for as long as
                      the block's host pointer, size and sub-chunk boundaries
                      stay the same (setting the mode again forgets this). No
                      extra copies are made.
   A host block without a device mapping is moved by the copy engines. Every
   mode gives identical bytes. Default: LST_COPY_AUTO both ways. On GB300 the
   copy engines give the fastest pipeline on pinned memory they move at the
   link rate (the copy kernels compete with the update kernel for the SMs);
   on the shared hosts measured here, the copy engines move parts of some
   pinned allocations at a few GB/s for their whole lifetime, and the copy
   kernel moved such parts faster. lst_stream_copy_choice reports what AUTO
   decided. LST_ERR_INVALID_ARG for another value. */
typedef enum { LST_COPY_ENGINE = 0, LST_COPY_SM = 1, LST_COPY_AUTO = 2 } lst_copy_mode;
LST_API lst_status lst_layout_set_stream_copy(lst_layout* layout, int32_t h2d_mode, int32_t d2h_mode);

/* What LST_COPY_AUTO has learned about block `block` of this layout:
   measured = 1 once a streamed step under LST_COPY_AUTO has timed the
   block's copy-engine copies (for its current host pointer); chunks = its
   sub-chunks in that step; kernel_in_chunks / kernel_out_chunks = how many of
   them later steps move with the copy kernel (0 under LST_COPY_ENGINE, all
   under LST_COPY_SM); and the slowest and fastest rates of its copy-engine
   sub-chunk copies of 4 MB or more timed each way (GB/s, 0 where none).
   Host only.
   Errors: LST_ERR_INVALID_ARG (null layout or out, block out of range). */
typedef struct lst_copy_choice {
  int32_t measured;
  int32_t chunks;
  int32_t kernel_in_chunks, kernel_out_chunks;
  double engine_h2d_gbs_min, engine_h2d_gbs_max;
  double engine_d2h_gbs_min, engine_d2h_gbs_max;
} lst_copy_choice;
LST_API lst_status lst_stream_copy_choice(const lst_layout* layout, int64_t block, lst_copy_choice* out);

/* The last streamed step on this layout that completed (lst_stream_step and
   its variants, including those lst_store_step runs): steps_completed counts
   them; h2d_bytes / d2h_bytes are the bytes it moved each way; chunks is its
   sub-chunk count and kernel_in_chunks / kernel_out_chunks how many of them
   the copy kernel moved; wall_ms is the host time from the call's first
   enqueue to the completion it observed. Under LST_COPY_AUTO (timed = 1)
   h2d_busy_ms / d2h_busy_ms are the summed durations of its copies each way
   (events on the copy streams): with the link busy in both directions at
   once, their sum exceeds wall_ms; 0 when not timed. All zero before the
   first completed step. Host only. Errors: LST_ERR_INVALID_ARG (null). */
typedef struct lst_stream_stats {
  int64_t steps_completed;
  int64_t h2d_bytes, d2h_bytes;
  int32_t chunks, kernel_in_chunks, kernel_out_chunks, timed;
  double wall_ms, h2d_busy_ms, d2h_busy_ms;
} lst_stream_stats;
LST_API lst_status lst_stream_last_stats(const lst_layout* layout, lst_stream_stats* out);

/* ------------------------------------------------------------------------
 * Device-resident step.
 * ------------------------------------------------------------------------ */

/* One AdamW step over every block, all blocks resident in device memory.
   dev_blocks: n_layers device pointers, one per block, each 16-byte aligned
   (null allowed only for a zero-byte block); the array itself is host memory
   and is read during the call only.
   cuda_stream: a cudaStream_t (null = the legacy default stream). The call
   enqueues one kernel launch per 128 blocks on that stream and returns; the
   update is complete when the stream reaches that point.
   Errors: LST_ERR_INVALID_ARG (null layout/hparams/dev_blocks, hparams outside
   their domain), LST_ERR_ALIGNMENT, LST_ERR_CUDA (launch failure). Validation
   happens before any CUDA call. */
LST_API lst_status lst_adamw_step(const lst_layout* layout, void* const* dev_blocks,
                          const lst_adamw_hparams* hparams, void* cuda_stream);

/* One SGD step, W += (-lr*g), over every block (m and v untouched; in the
   mixed layout the master moves and W is re-derived). As lst_adamw_step. */
LST_API lst_status lst_sgd_step(const lst_layout* layout, void* const* dev_blocks, float lr,
                        void* cuda_stream);

/* ------------------------------------------------------------------------
 * Per-block options: step counters, locked blocks, gradient magnitude.
 * ("Training 70B Models on Consumer Hardware", section "Progressive Layer
 * Locking": a layer whose gradient magnitude falls below a threshold is
 * locked - no update and no I/O for it; and the note under "The Math": with
 * locking, per-layer step counters keep Adam's bias correction exact.)
 * ------------------------------------------------------------------------ */
typedef struct lst_step_options {
  /* Host array [n_layers] of per-block step counters t_i >= 1 for the bias
     corrections, or NULL: hparams->step for every block. */
  const int64_t* block_steps;
  /* Host array [n_layers]; a nonzero entry marks a locked block: it is neither
     read nor written (and, in the streamed step, not transferred). NULL: none. */
  const uint8_t* skip;
  /* DEVICE array [n_layers] of doubles, or NULL. When given, every block that
     is not skipped receives sum(g^2) over its elements (its squared gradient
     L2 norm), computed in the same pass as the update: per group of 8
     elements in fp32, accumulated in an fp32 pair that recovers each
     addition's rounding error exactly, then in fp64, in a fixed order
     (deterministic for a given device). Entries of skipped blocks are left
     untouched. Written asynchronously on the call's stream (by a second,
     small launch after the update). */
  double* grad_sq;
  /* DEVICE scratch of lst_workspace_bytes() bytes, 256-byte aligned; required
     when grad_sq is given. Calls that share a workspace must not overlap on
     the GPU. Its contents on entry do not matter. */
  void* workspace;
} lst_step_options;

/* Bytes of device workspace the sum-of-squares reduction needs (a constant:
   one 8-byte partial sum per CTA, up to 1024 CTAs, and per block of one
   launch, up to 128 blocks, after a reserved 256-byte header). */
LST_API int64_t lst_workspace_bytes(void);

/* lst_adamw_step with per-block options (opts may be NULL). Results of a
   block with step t_i are bit-identical to lst_adamw_step on that block alone
   with step = t_i. Errors as lst_adamw_step, plus LST_ERR_INVALID_ARG for a
   block step < 1 or grad_sq without workspace, LST_ERR_ALIGNMENT for a
   misaligned workspace or grad_sq. */
LST_API lst_status lst_adamw_step_ex(const lst_layout* layout, void* const* dev_blocks,
                                     const lst_adamw_hparams* hparams, const lst_step_options* opts,
                                     void* cuda_stream);

/* ------------------------------------------------------------------------
 * For callers that cannot allocate device memory. The pages have no
 * counterpart to this call; it exists so that the library can be used where
 * device allocation is not available to the caller.
 * ------------------------------------------------------------------------ */

/* lst_adamw_step_ex, with the scratch of its sum-of-squares reduction taken
   from memory the library holds itself instead of a caller's workspace.
   It is meant for callers that cannot allocate device memory when they step
   the optimizer: a plugin running inside an application whose device memory
   belongs to another allocator, a training loop that has handed all device
   memory to a framework's caching pool, or code that must not allocate once
   it is running.
   The scratch is one static device array of lst_workspace_bytes() bytes
   (1 MiB + 256 bytes). Every GPU that loads the library's device code holds
   it until the process exits. It holds the partial sums of one launch (128
   blocks); a step over more blocks runs as several launches in order on the
   one stream, which reuse the array one after the other, so there is no limit
   on the number of blocks. Without grad_sq no scratch is used.
   The first call on a device that passes grad_sq looks up the array's device
   address (cudaGetSymbolAddress) with that device current; make that first
   call before any stream capture. The address is kept for the process's
   lifetime: the call assumes the runtime's primary context on each device and
   no cudaDeviceReset after that first call. The call allocates nothing: no
   cudaMalloc, no cudaFree, no allocating library routine.
   All calls share the one array, which keeps the last call's contents;
   nothing in it needs to start at any value. Calls whose
   work overlaps on the GPU (streams with no ordering between them) race on
   the array: order them, or use lst_adamw_step_ex with separate workspaces.
   block_steps, skip: host arrays of n_layers entries, or NULL; grad_sq: a
   device array of n_layers doubles, or NULL. Results are those of
   lst_adamw_step_ex with the same arguments. Errors as lst_adamw_step_ex. */
LST_API lst_status lst_adamw_step_ex_noalloc(const lst_layout* layout, void* const* dev_blocks,
                                             const lst_adamw_hparams* hparams, const int64_t* block_steps,
                                             const uint8_t* skip, double* grad_sq, void* cuda_stream);

/* ------------------------------------------------------------------------
 * Streamed step ("MegaTrain" summary page: host memory is the authoritative
 * store; StreamIn over a weight stream, compute, offload over a second copy
 * stream; two buffers ping-pong; events weights-ready, update-done and
 * buffer-free; no host-side barrier).
 * ------------------------------------------------------------------------ */

/* One AdamW step over every block, blocks in pinned host memory.
   host_blocks: n_layers pointers to page-locked host memory (cudaHostAlloc,
   cudaHostRegister or lst_host_alloc), each 4096-byte aligned and at least
   the block's size. dev_buf0, dev_buf1: two device buffers, each 256-byte
   aligned and at least max_block_bytes (lst_layout_info) long; the k-th
   block transferred is staged in buffer k & 1, at the block's own offsets.
   For each block, in sub-chunks of the layout's stream chunk size: the input
   prefix is copied host -> device on a copy stream, the update runs on a
   compute stream, and the output suffix is copied device -> host on a second
   copy stream; the streams wait only on events. The copies are copy-engine
   transfers or, per lst_layout_set_stream_copy, an SM copy kernel on the same
   copy stream. Results are bit-identical to lst_adamw_step on the same data.
   Synchronous: returns when all copies back to the host blocks are complete,
   or with LST_ERR_TIMEOUT once timeout_ms has passed (timeout_ms <= 0: no
   deadline); in that case work
   may still be in flight and the caller must synchronize the device before
   touching or freeing host_blocks or the device buffers. The device buffers
   must not be in use by other work during the call.
   Errors: LST_ERR_INVALID_ARG, LST_ERR_ALIGNMENT, LST_ERR_NOT_PINNED,
   LST_ERR_CUDA (after draining what was already enqueued; blocks before the
   failure point may already hold updated state, so the step must be treated
   as failed as a whole), LST_ERR_TIMEOUT. */
LST_API lst_status lst_stream_step(const lst_layout* layout, void* const* host_blocks, void* dev_buf0,
                           void* dev_buf1, const lst_adamw_hparams* hparams, int64_t timeout_ms);

/* lst_stream_step with per-block options (opts may be NULL). A locked block
   (skip) is not transferred in either direction and not updated. grad_sq is
   a device array; it is complete when the call returns LST_OK. Results of
   every block are bit-identical to lst_adamw_step_ex on the same data. */
LST_API lst_status lst_stream_step_ex(const lst_layout* layout, void* const* host_blocks, void* dev_buf0,
                                      void* dev_buf1, const lst_adamw_hparams* hparams,
                                      const lst_step_options* opts, int64_t timeout_ms);

/* The streamed step for gradients that are already on the device, as a
   backward pass leaves them. The "MegaTrain" page offloads gradients to the
   host after backward (three-stream execution: a gradient stream for the
   device-to-host offload) because its optimizer runs on the CPU; with the
   update on the GPU the gradient never has to leave the device, so only the
   state crosses the link inbound (L12: W|m|v, 10 B/param; L16M:
   master|m|v, 12 B/param; L16F: W|m|v, 12 B/param), and the outbound bytes
   are unchanged.
   dev_grads: n_layers device pointers (16-byte aligned; ignored for skipped
   or empty blocks), each to a block's gradient laid out as its G segment:
   padded_elems elements of the G type (bf16, or fp32 for LST_L16_FP32), with
   zeros in the padding. The G segments of the host blocks are neither read
   nor written. The gradients must be complete when the call is made: the
   call does not wait on other streams. opts may be NULL. Otherwise as
   lst_stream_step_ex; results are bit-identical to it when the host G
   segments hold the same gradient. */
LST_API lst_status lst_stream_step_devgrad(const lst_layout* layout, void* const* host_blocks,
                                           const void* const* dev_grads, void* dev_buf0, void* dev_buf1,
                                           const lst_adamw_hparams* hparams, const lst_step_options* opts,
                                           int64_t timeout_ms);

/* The device-gradient streamed step overlapped with the backward pass that
   produces the gradients ("MegaTrain" summary page, three-stream execution:
   a Backward-Done event per layer releases that layer's gradient). Block i's
   update waits, on the device, for grad_ready[i]: a cudaEvent_t that the
   producer recorded on its own stream after writing dev_grads[i]. The state
   of a block is copied in without waiting for it, so block i's state streams
   in, is updated and streams out while gradients of later blocks in `order`
   are still being produced; the host never waits for the producer.
   grad_ready: host array of n_layers cudaEvent_t values (as void*); a NULL
   entry means that block's gradient is already complete. Each event must
   have been recorded before this call: the wait binds to its latest record
   at the time of the call. The events are not modified.
   order: host array holding a permutation of 0..n_layers-1, the order in
   which blocks are transferred and updated (a backward pass completes its
   layers last to first: order = n_layers-1, ..., 0), or NULL for index order.
   Otherwise as lst_stream_step_devgrad; results are bit-identical to it.
   Errors as lst_stream_step_devgrad, plus LST_ERR_INVALID_ARG when order is
   not a permutation, and LST_ERR_CUDA when a wait on an event fails. */
LST_API lst_status lst_stream_step_devgrad_events(const lst_layout* layout, void* const* host_blocks,
                                                  const void* const* dev_grads, void* const* grad_ready,
                                                  const int64_t* order, void* dev_buf0, void* dev_buf1,
                                                  const lst_adamw_hparams* hparams, const lst_step_options* opts,
                                                  int64_t timeout_ms);

/* One AdamW step with the update kernel reading and writing the pinned host
   blocks in place over the host link (NVLink-C2C on Grace systems): no device
   buffers, no copy engines. This is the zero-copy staging the "MegaTrain"
   summary page mentions for its 4 KB-aligned blocks, taken to its end: the
   kernel is the only consumer of the staged bytes, so it may as well read
   them where they are. Results are bit-identical to lst_adamw_step.
   host_blocks: n_layers pointers to page-locked host memory that is mapped
   into the device address space (lst_host_alloc, cudaHostAlloc, or
   cudaHostRegister with cudaHostRegisterMapped), each 4096-byte aligned.
   Asynchronous on cuda_stream, like lst_adamw_step; the host must not touch
   the blocks until the stream has passed the step.
   Errors: LST_ERR_INVALID_ARG, LST_ERR_ALIGNMENT, LST_ERR_NOT_PINNED (not
   pinned, or not mapped), LST_ERR_CUDA. */
LST_API lst_status lst_zero_copy_step(const lst_layout* layout, void* const* host_blocks,
                                      const lst_adamw_hparams* hparams, void* cuda_stream);

/* ------------------------------------------------------------------------
 * File-backed block store: the tier under host memory. ("Training 70B Models
 * on Consumer Hardware": model state in per-layer files on an SSD,
 * pre-allocated with fallocate, flushed after each update, and - its safety
 * note - a persisted step counter and atomic writes or shadow copies so that a
 * crash cannot corrupt state. The "MegaTrain" summary page: SSDs as the next
 * tier below host memory.)
 * A store is a directory with one file per block: a 4096-byte header (magic,
 * the layout's fingerprint for that block, the block's step counter, a header
 * checksum) followed by the block's bytes. Files are read and written with
 * direct I/O when the file system allows it. A block is committed by writing
 * a shadow file, flushing it (fsync), renaming it over the block file and
 * flushing the directory, so after a crash every block is at its old or its
 * new step, never torn. The layout must outlive the store.
 * ------------------------------------------------------------------------ */

/* Create (or overwrite) a store in directory dir (created if missing, one
   level) with every block at step counter `step` (>= 0). host_blocks: NULL
   (blocks start zeroed) or n_layers host pointers, each 4096-byte aligned (a
   NULL entry gives a zeroed block). Errors: LST_ERR_INVALID_ARG,
   LST_ERR_ALIGNMENT, LST_ERR_IO, LST_ERR_OOM. */
LST_API lst_status lst_store_create(const lst_layout* layout, const char* dir, void* const* host_blocks,
                                    int64_t step, lst_store** out);

/* Open an existing store. Every block file's header must match the layout
   (LST_ERR_INVALID_ARG otherwise; LST_ERR_IO for a missing or damaged file).
   A shadow file left by an interrupted commit is discarded: the block file
   still holds the committed state. */
LST_API lst_status lst_store_open(const lst_layout* layout, const char* dir, lst_store** out);

/* Release the handle (the files stay). NULL is ignored. */
LST_API void lst_store_close(lst_store* store);

/* The step counter a block was last committed with. */
LST_API lst_status lst_store_block_step(const lst_store* store, int64_t layer, int64_t* step);

/* Read a block's bytes into host memory (4096-byte aligned, at least the
   block's size), e.g. to inspect it or to write a gradient into its G
   segment. */
LST_API lst_status lst_store_read(const lst_store* store, int64_t layer, void* host_dst);

/* Commit a block's bytes from host memory (4096-byte aligned) with step
   counter `step` (>= 0), atomically as described above. */
LST_API lst_status lst_store_write(lst_store* store, int64_t layer, const void* host_src, int64_t step);

/* One AdamW step (hparams->step = t >= 1) over every block of the store whose
   committed step counter is t - 1: read it from its file, update it with the
   streamed step (lst_stream_step_ex on that block, through dev_buf0/dev_buf1),
   commit it with step counter t. Blocks already at step t or beyond are
   skipped, so a step that failed or was interrupted is completed by calling it
   again with the same arguments: each block is updated exactly once. A block
   below t - 1 has missed a step: LST_ERR_INVALID_ARG before anything is done.
   The gradient is whatever the block file's G segment holds.
   staging: three pinned host buffers (lst_host_alloc), each 4096-byte aligned
   and at least max_block_bytes long; reading block k+1, updating block k and
   committing block k-1 overlap on them. dev_buf0/1 and timeout_ms as in
   lst_stream_step (the deadline applies per block). Synchronous. Errors: those
   of lst_stream_step, plus LST_ERR_IO; after an error, blocks committed so far
   are at step t and the others at t - 1. */
LST_API lst_status lst_store_step(lst_store* store, void* const* staging, void* dev_buf0, void* dev_buf1,
                                  const lst_adamw_hparams* hparams, int64_t timeout_ms);

/* ------------------------------------------------------------------------
 * Utilities.
 * ------------------------------------------------------------------------ */

/* Page-locked host memory: page-aligned (at least 4096 bytes) anonymous
   memory registered with CUDA as mapped and portable, so a device kernel may
   also address it directly. Free with lst_host_free (LST_ERR_INVALID_ARG for
   a pointer that did not come from lst_host_alloc). LST_ERR_OOM if the memory
   cannot be reserved or pinned. */
LST_API lst_status lst_host_alloc(int64_t bytes, void** out);
LST_API lst_status lst_host_free(void* ptr);

/* Static description of a status code. */
LST_API const char* lst_status_string(lst_status status);

/* Text of the last error raised on the calling thread ("" if none). */
LST_API const char* lst_last_error(void);

/* Test hook (host-side fault injection; no device fault is ever caused).
   kind 0: clear. kind 1: the k-th asynchronous enqueue (copy, launch, event
   record or wait; counted from 1 within each later lst_stream_step call)
   reports a failure instead of being issued. kind 2: lst_stream_step never
   observes completion, so it returns LST_ERR_TIMEOUT at its deadline (after
   which it still drains its own work before returning). kind 3: committing
   block k-1 of a store (lst_store_write, lst_store_step) fails after its
   shadow file is written and flushed, before the rename, as a crash there
   would. kind 4: LST_COPY_AUTO sees the copy-engine sub-chunk copies of
   every k-th block (blocks 0, k, 2k, ...; k >= 1) as 100x slower than they
   were (nothing is slowed down), as on a host whose pinned memory the copy
   engines move slowly in places. */
LST_API lst_status lst_test_inject(int32_t kind, int64_t k);

#ifdef __cplusplus
}
#endif

#endif /* LST_H */
