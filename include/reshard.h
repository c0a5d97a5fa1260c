/*
 * reshard.h -- C ABI of the single-GPU DTensor -> DTensor reshard executor (libreshard.so).
 *
 * The operation is the Reshard collective: move a tensor's values from a source distribution
 * (M local shards over a device mesh with Shard/Replicate placements) to a destination
 * distribution (N local shards, possibly replicated), sending only the regions where source
 * and destination shards overlap and reading each region once even when several destination
 * replicas need it. Definitions used below:
 *  - news article on NVIDIA's Reshard collective, sections "Recasting refit as a
 *    DTensor-to-DTensor transfer" and "The Reshard collective";
 *  - NeMo-RL design doc "NCCL Reshard Refit (Experimental)": "Execution Flow: Setup Time"
 *    (global shape, dtype, MeshInfo, Shard/Replicate placements), "xferdtensor Transports"
 *    (exact overlaps, each destination region moved once, fan-out to replicas, the stream
 *    argument), "Enabling It" (BF16 -> MXFP8 on the receive side, one ValueError listing every
 *    violation);
 *  - "NeMo-RL: Optimizing Non-Colocated Refit for Asynchronous RL", "Optimization #2"
 *    (coalesce many tensors into one call; pack into contiguous messages).
 *
 * In the single-process calls all M source and N destination shards are buffers reachable from
 * ONE GPU, so "sending" a region is a device copy. The work is split into a host-side plan
 * (built once, cached: "descriptor caching" in the ModelExpress reshard PR) and an asynchronous
 * execute. When the shards are spread over several processes (one GPU each), every process runs
 * its share of the plan (reshard_plan_partition): local copies and packing of outgoing messages,
 * the listed point-to-point transfers (moved by the caller's communication library), unpacking.
 *
 * Conventions
 *  - All sizes, offsets and strides are in ELEMENTS of the tensor's dtype unless named _bytes.
 *  - Ranks are numbered row-major over mesh coordinates. mesh.ranks, when given, maps the
 *    row-major position to the index of that rank's pointer in the execute pointer arrays
 *    (a permutation of 0..n-1); NULL means the identity.
 *  - Uneven splits follow torch.chunk: chunk = ceil(L / n), rank i holds
 *    [min(i chunk, L), min((i + 1) chunk, L)); trailing ranks may hold nothing.
 *  - Several mesh dims sharding one tensor dim split in mesh-dim order (nested).
 *  - Errors: every call returns 0 (RESHARD_OK) or a negative RESHARD_ERR_* code, and
 *    reshard_last_error() then describes it. Validation lists EVERY violation it finds, one
 *    per line, and fails closed: no plan is returned.
 *  - Thread safety: plans are not locked. Calls on different plans may run concurrently; calls
 *    on one plan must be serialised by the caller. The error text is per thread.
 */
#ifndef RESHARD_H
#define RESHARD_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define RESHARD_MAX_DIMS 4      /* tensor dims */
#define RESHARD_MAX_MESH_DIMS 4 /* device-mesh dims */

/* return codes */
#define RESHARD_OK 0
#define RESHARD_ERR_INVALID_ARG (-1) /* malformed spec, pointer or argument */
#define RESHARD_ERR_UNSUPPORTED (-2) /* well formed but outside what the executor handles */
#define RESHARD_ERR_CUDA (-3)        /* a CUDA runtime call failed (message has the name) */
#define RESHARD_ERR_OOM (-4)         /* host or device allocation failed */
#define RESHARD_ERR_COVERAGE (-5)    /* the plan would leave destination elements unwritten */

/* placement kinds (DTensor Shard(dim) / Replicate()) */
#define RESHARD_REPLICATE 0
#define RESHARD_SHARD 1

/* element types. Copies move bytes, so every type is bit-exact; only BF16 can be quantized. */
#define RESHARD_U8 0
#define RESHARD_BF16 1
#define RESHARD_F16 2
#define RESHARD_F32 3
#define RESHARD_I32 4
#define RESHARD_I64 5

/* execute modes */
#define RESHARD_DIRECT 0 /* one pass: source regions straight into every destination replica */
#define RESHARD_PACKED 1 /* pack per-(source, destination group) messages, then unpack them */

/* receive-side quantization */
#define RESHARD_QUANT_NONE 0
#define RESHARD_QUANT_MXFP8 1 /* BF16 -> E4M3 bytes + one E8M0 scale byte per 32 elements */

/* partitioned plans (multi-process exchange) */
#define RESHARD_STRIPED 1  /* reshard_plan_partition flag: striped two-phase receive */
#define RESHARD_SEND 0     /* reshard_transfer_t.dir */
#define RESHARD_RECV 1
#define RESHARD_SEND_BUF 0 /* reshard_transfer_t.buf */
#define RESHARD_RECV_BUF 1

/* Opaque CUDA stream; pass a cudaStream_t (NULL = the legacy default stream). */
struct CUstream_st;
typedef struct CUstream_st *reshard_stream_t;

/* Device mesh ("MeshInfo"): an ndim-dimensional grid of ranks. */
typedef struct {
  int ndim;              /* 1..RESHARD_MAX_MESH_DIMS */
  const int64_t *shape;  /* ndim extents, each >= 1 */
  const int32_t *ranks;  /* prod(shape) pointer indices (a permutation), or NULL = identity */
} reshard_mesh_t;

/* One placement per mesh dim. */
typedef struct {
  int kind; /* RESHARD_SHARD or RESHARD_REPLICATE */
  int dim;  /* sharded tensor dim for RESHARD_SHARD; ignored for RESHARD_REPLICATE */
} reshard_placement_t;

/* Where a rank's local shard sits in its buffer ("DTensorRef" local tensor, or a slice of a
 * fused parameter such as gate_up: design doc, "Execution Flow: Setup Time").
 * The element at local index i is at buffer element offset_elems + sum_d i[d] * strides[d].
 * Strides are non-negative. A destination view must not map two elements to one offset: taken
 * by increasing stride, each dim's stride must exceed the span of the dims below it (dense,
 * padded, transposed and interleaved layouts all do); the plan refuses one that does not
 * (INVALID_ARG naming the view). Source views are only read and may alias. When the source and the
 * destination of a region are contiguous along the same dim, the region is a strided copy;
 * when they are contiguous along different dims (a transposed layout on one side, e.g. a
 * destination that keeps W^T), the region goes through the TMA transposing kernel; with no
 * contiguous dim at all it is copied element by element. */
typedef struct {
  int64_t offset_elems;          /* >= 0 */
  const int64_t *strides_elems;  /* ndim strides (>= 0); NULL = dense row-major */
  int64_t capacity_elems;        /* elements the buffer holds (bounds check); 0 = not checked */
} reshard_view_t;

/* One tensor: the DTensor description on both sides. */
typedef struct {
  int ndim;                      /* 1..RESHARD_MAX_DIMS */
  const int64_t *global_shape;   /* ndim extents, each >= 0 */
  int dtype;                     /* RESHARD_U8 .. RESHARD_I64 */
  reshard_mesh_t src_mesh;
  const reshard_placement_t *src_pl;  /* src_mesh.ndim placements */
  const reshard_view_t *src_views;    /* prod(src_mesh.shape) views (pointer-index order) or NULL */
  reshard_mesh_t dst_mesh;
  const reshard_placement_t *dst_pl;
  const reshard_view_t *dst_views;
} reshard_tensor_spec_t;

typedef struct reshard_plan reshard_plan_t;

/* Plan statistics (the byte accounting of the ModelExpress reshard PR, "MoE Qwen3-30B-A3B:
 * expert coverage": planned wire bytes vs engine bytes, exact descriptor count). */
typedef struct {
  int64_t n_tensors;
  int64_t regions;            /* (source, destination group) overlaps, each moved once */
  int64_t items;              /* device work items of the direct mode */
  int64_t dst_groups;         /* destination replica groups (distinct destination boxes) */
  int64_t messages;           /* (source rank, destination group) pairs with data */
  int64_t bytes_read;         /* source bytes read per direct execute */
  int64_t bytes_written;      /* destination bytes written per execute (unquantized) */
  int64_t wire_bytes;         /* bytes a wire transport would carry: each region once */
  int64_t message_bytes;      /* packed-mode workspace: messages with 16-byte aligned regions */
  int64_t gather_bcast_bytes; /* all-gather + broadcast payload for comparison: 2 x tensor bytes */
  int64_t global_bytes;       /* sum of global tensor bytes */
  int64_t last_launches;      /* kernel launches enqueued by the plan's last execute */
  int64_t last_aligned_items; /* copy items of its last pass run by the aligned walker ... */
  int64_t last_general_items; /* ... and by the general (unaligned-capable) walker */
  int64_t last_rows_kernel;   /* 1 if those ran in its many-short-rows build
                                 (reshard_copy_rows_kernel), 0 if in reshard_copy_kernel */
  /* the message buffers of reshard_execute_pack / _unpack: message_bytes (above) is the send
   * buffer's size, recv_bytes the receive buffer's (equal for an unpartitioned plan) */
  int64_t recv_bytes;
  int64_t rank;               /* the process a partitioned plan is for; -1 if unpartitioned */
  int64_t world;              /* processes of the partition; 0 if unpartitioned */
  int64_t transfers;          /* point-to-point operations of this rank, both phases */
  int64_t sent_bytes;         /* bytes this rank sends in phase 1 (its own sources' messages) */
  int64_t forwarded_bytes;    /* bytes this rank forwards in phase 2 (stripes it received) */
  int64_t local_bytes;        /* source bytes this rank copies to its own destinations directly */
  int64_t last_staged_items;  /* copy items of the last execute's last pass run by the bulk-staged
                                 kernel (reshard_copy_staged_kernel: misaligned rows < 4 KiB) */
  int64_t gather_items;       /* pair items of all passes (reshard_plan_items sets 6-8): destination
                                 rows of two source pieces (direct, unpack) and source rows into two
                                 message blocks (pack) */
  int64_t last_gather_items;  /* pair items run by the last execute (reshard_copy_gather_kernel,
                                 reshard_copy_scatter_kernel) */
} reshard_stats_t;

/* One point-to-point transfer of a partitioned plan (see reshard_plan_transfers). */
typedef struct {
  int32_t peer;   /* the process at the other end */
  int32_t dir;    /* RESHARD_SEND or RESHARD_RECV */
  int32_t buf;    /* this rank's buffer: RESHARD_SEND_BUF or RESHARD_RECV_BUF */
  int32_t phase;  /* 1 or 2 */
  int64_t offset; /* byte offset in that buffer (a multiple of 16) */
  int64_t bytes;  /* a multiple of 16, > 0 */
} reshard_transfer_t;

/*
 * reshard_plan_create -- plan one tensor's reshard (host only; touches no GPU).
 * spec: the tensor; read during the call only.  out: receives the plan (caller destroys it).
 * Steps: every rank's box by the chunk rule; replica groups of identical boxes on each side;
 * per-dim intersection of every source group with every destination group; one source per
 * region (the lowest pointer index of the source group); work items for the device.
 * Errors: INVALID_ARG / UNSUPPORTED listing every violation; OOM.
 */
int reshard_plan_create(const reshard_tensor_spec_t *spec, reshard_plan_t **out);

/*
 * reshard_plan_batch -- one plan over n_tensors tensors, executed by one launch per pass.
 * Pointer arrays of the execute are the per-tensor arrays concatenated in spec order: tensor t
 * owns prod(src_mesh.shape) consecutive source pointers and prod(dst_mesh.shape) consecutive
 * destination pointers (two per rank under MXFP8, see reshard_execute).
 */
int reshard_plan_batch(const reshard_tensor_spec_t *specs, int n_tensors, reshard_plan_t **out);

/*
 * reshard_plan_blockwise_fp8 -- plan FP8 weights together with their blockwise scales, the
 * blockwise-FP8 train <-> FP8 gen path of the design doc ("Enabling It"; the FP8 "_scale_inv"
 * siblings of "Design Overview"). specs: n_tensors FP8 weights (dtype RESHARD_U8, ndim >= 2).
 * For each, a scale tensor is derived: global shape with the last two dims ceil-divided by
 * block_rows / block_cols, dtype RESHARD_F32, the same meshes and placements, dense views.
 * The plan is a batch of 2 n_tensors tensors: the weights in spec order, then their scales in
 * the same order; pointer arrays follow that order (weights' pointers, then scales').
 * Every shard boundary of a weight along the two blocked dims must fall on a block boundary
 * (or at the tensor's end) on both sides, so that each scale shard is exactly the blocks of
 * its weight shard; otherwise UNSUPPORTED, listing the offending tensors and dims.
 */
int reshard_plan_blockwise_fp8(const reshard_tensor_spec_t *specs, int n_tensors, int64_t block_rows,
                               int64_t block_cols, reshard_plan_t **out);

/*
 * reshard_execute -- enqueue the reshard on `stream` and return (asynchronous).
 * src_ptrs / dst_ptrs: HOST arrays of pointers, caller-owned, laid out as above. A rank whose
 *   shard is empty may pass NULL. Each pointer is memory of the plan's device, managed memory,
 *   or page-locked host memory mapped into the device's address space (cudaHostAlloc,
 *   cudaMallocHost, cudaHostRegister). The kernels read and write host memory in place over
 *   the host link, so a host-to-host reshard needs no staging copies in device memory; the
 *   transposing regions then read it with plain loads instead of TMA. Pageable host memory
 *   and another device's memory are refused (INVALID_ARG, naming up to eight pointers); the
 *   check (cudaPointerGetAttributes per pointer) runs whenever the pointers change. Under RESHARD_QUANT_MXFP8 dst_ptrs holds two entries
 *   per destination rank: the E4M3 data buffer (1 byte per element, dense row-major of the
 *   local shape, at element offset offset_elems) and the E8M0 scale buffer (1 byte per 32
 *   elements, row-major [..., K_local / 32], at offset_elems / 32).
 * mode: RESHARD_DIRECT or RESHARD_PACKED.  quant: RESHARD_QUANT_NONE or RESHARD_QUANT_MXFP8
 *   (BF16 tensors only; every destination's last local dim and every region boundary along it
 *   a multiple of 32; dense destination views; otherwise UNSUPPORTED).
 * The first execute binds the plan to the current device and uploads its descriptor tables
 * (synchronous device allocations: do it outside stream capture); RESHARD_PACKED also
 * allocates the message workspace (stats.message_bytes) on first use. When the pointers differ
 * from the previous call's, the changed ones are checked, the pointer table is re-uploaded on
 * `stream`, the TMA tensor maps of transposing regions are re-encoded, and the copy items are
 * re-sorted on the host into those 16-byte aligned everywhere (run by the aligned walker),
 * misaligned items of rows shorter than 4 KiB in device memory (run by the bulk-staged kernel)
 * and the rest (run by the general walker), and the gather items (destination rows of two
 * source pieces, reshard_plan_items sets 6 and 8; run by the gather kernel in passes without
 * quantization) are resolved to absolute addresses and re-uploaded on `stream`: host work
 * proportional to the plan's items, none when the pointers repeat. Those uploads copy from the
 * plan's host tables, so an execute captured into a CUDA graph should repeat the pointers of an
 * execute made before the capture (it then enqueues kernel launches only).
 * Buffers must stay valid until the stream reaches the end of the work. Executes of one plan
 * on different streams that overlap in time race on its tables and workspace.
 * Errors: INVALID_ARG (NULL pointer of a shard the plan reads or writes, a pointer the device
 *   cannot dereference, plan bound to another device, a partitioned plan), UNSUPPORTED,
 *   CUDA (launch or copy failure), OOM. After an error the destinations are undefined.
 */
int reshard_execute(reshard_plan_t *plan, void *const *src_ptrs, void *const *dst_ptrs, int mode,
                    int quant, reshard_stream_t stream);

/*
 * reshard_execute_pack / reshard_execute_unpack -- the two passes of the packed mode with
 * message buffers owned by the caller, so that a transport can move the messages in between
 * ("NeMo-RL: Optimizing Non-Colocated Refit for Asynchronous RL", "Optimization #2": coalesce
 * many tensors and pack them into contiguous buffers that move in few large transfers).
 * pack reads the sources and writes send_buf (stats.message_bytes bytes). On a partitioned plan
 *   (reshard_plan_partition) it also copies every region whose source and destination are both
 *   on this rank straight into the destination (quantized under RESHARD_QUANT_MXFP8: dst_ptrs
 *   then holds data/scale pairs as in reshard_execute); on an unpartitioned plan dst_ptrs may be
 *   NULL and quant must be RESHARD_QUANT_NONE.
 * unpack reads recv_buf (stats.recv_bytes bytes) and writes the destinations (quantizing under
 *   RESHARD_QUANT_MXFP8, with the same constraints as reshard_execute).
 * Message layout: regions in plan order, each starting on a 16-byte boundary; on an
 *   unpartitioned plan it is the packed mode's (messages per (source rank, destination group),
 *   both buffers the same size; they may be one buffer), so pack then unpack equals
 *   reshard_execute(RESHARD_PACKED) with a caller-owned workspace.
 * Buffers: device memory of the plan's device or page-locked host memory (as in
 *   reshard_execute), 16-byte aligned, valid until the stream reaches the end of the work. Both
 *   calls are asynchronous on `stream`; pointer arrays as in reshard_execute (on a partitioned
 *   plan only this rank's entries are read; the others may be NULL).
 * Errors as reshard_execute; INVALID_ARG also for a buffer that is NULL or not 16-byte aligned
 *   while the plan has messages.
 */
int reshard_execute_pack(reshard_plan_t *plan, void *const *src_ptrs, void *const *dst_ptrs, void *send_buf,
                         int quant, reshard_stream_t stream);
int reshard_execute_unpack(reshard_plan_t *plan, const void *recv_buf, void *const *dst_ptrs, int quant,
                           reshard_stream_t stream);

/*
 * reshard_plan_partition -- the share of `plan` that one process runs when the shards live on
 * different processes (one GPU each) of a process group: the multi-GPU form of the Reshard
 * collective (NeMo-RL design doc "NCCL Reshard Refit (Experimental)", "xferdtensor Transports":
 * batched point-to-point transfers, receives striped across destination replicas, then spread
 * inside each replica group; news article on NVIDIA's Reshard collective, "How NCCL M2N Reshard
 * maximizes network bandwidth": each replica group pulls a byte over the network once and its
 * members exchange their stripes over NVLink).
 * src_owner[i], dst_owner[j]: the process (0 .. world-1) that holds source pointer i and
 *   destination pointer j of `plan` (flat pointer-array order, as in reshard_execute).
 * rank: the process to plan for. flags: 0 or RESHARD_STRIPED.
 * Source choice: each region is sent by one holder of its source box; a holder on a process
 *   that also holds a destination of the region is preferred (that copy stays local), otherwise
 *   the holders take regions in turn. Messages: one per (sending process, set of other processes
 *   receiving), holding the regions of every tensor it carries in plan order, 16-byte aligned;
 *   the send buffer holds this rank's outgoing messages, the receive buffer its incoming ones,
 *   each ordered by (sender, receivers).
 * Transfers: without RESHARD_STRIPED each receiver gets every message whole from its sender
 *   (phase 1). With it a message is cut into one 16-byte aligned stripe per receiver; the
 *   sender sends stripe k to the k-th receiver (phase 1) and each receiver forwards its stripe to
 *   the message's other receivers (phase 2), so each message byte leaves the sender once.
 * Use: reshard_execute_pack (local copies, outgoing messages), then every transfer of phase 1,
 *   then of phase 2 (reshard_plan_transfers), then reshard_execute_unpack. The result is a new
 *   host-only plan; `plan` is not modified and may be destroyed. A partitioned plan cannot run
 *   through reshard_execute or reshard_execute_static, and cannot be partitioned again.
 * Errors: INVALID_ARG (NULL arguments, world < 1, rank or an owner out of range, a partitioned
 *   plan, unknown flags); OOM.
 */
int reshard_plan_partition(const reshard_plan_t *plan, const int32_t *src_owner, const int32_t *dst_owner, int world,
                           int rank, int flags, reshard_plan_t **out);

/*
 * reshard_plan_transfers -- the point-to-point transfers of a partitioned plan's rank in one
 * phase (1 or 2), in posting order: for every pair of processes the sender's sends and the
 * receiver's receives of a phase are listed in the same order with the same sizes, so that
 * in-order matching (MPI, NCCL and gloo point-to-point semantics) pairs them correctly. All of
 * phase 1 must complete before phase 2 starts (phase 2 sends read stripes received in phase
 * 1). Up to cap entries go to `out` (may be NULL); *n_out gets the count. Empty for an
 * unpartitioned plan.
 */
int reshard_plan_transfers(const reshard_plan_t *plan, int phase, int64_t cap, reshard_transfer_t *out,
                           int64_t *n_out);

/*
 * reshard_execute_static -- the direct-mode reshard (quant none) without any device allocation.
 * The pages have no counterpart to this call; it exists for callers that cannot let a library
 * allocate device memory during a refit: an inference engine that has reserved nearly all of
 * the GPU for its KV cache, or a framework whose own caching allocator owns the device heap,
 * where cudaMalloc could fail for lack of memory and cudaMalloc/cudaFree would synchronize the
 * device and stall work already running.
 * The plan's descriptor tables and the pointer table are copied (cudaMemcpyAsync on `stream`,
 * from pageable memory, staged before the call returns) into one file-scope device array of
 * RESHARD_STATIC_SCRATCH_BYTES bytes that the library image holds on every GPU that loads it,
 * until the process exits; then the same copy kernel as reshard_execute runs from there.
 * Set-up: every call, an empty plan's included, looks the array's device address up on the
 * current device (cudaGetSymbolAddress, once per device; it also loads the library's device code
 * there, which is when the array is reserved under lazy module loading, the CUDA default). So the
 * first call on a device does that set-up: make it before any stream capture, and early (an empty
 * plan will do) if the rest of device memory is about to be reserved by the caller.
 * Calls on one device share the array and it keeps the last call's contents (nothing in it needs
 * to start at zero): calls that overlap on the GPU race, so serialise them (for example, all on
 * one stream).
 * Arguments as in reshard_execute (one destination pointer per rank). The pointers are checked
 * as reshard_execute checks them (cudaPointerGetAttributes, a host-side query that allocates
 * nothing): pageable host memory and other devices' memory are refused with INVALID_ARG; the last
 * accepted pointer set of each device is remembered, so repeating it skips the queries. The plan is
 * only read and is not bound to a device; plans with transposing regions are UNSUPPORTED here
 * (their tensor maps live with the plan), and partitioned plans INVALID_ARG.
 * Errors: INVALID_ARG (NULL plan, a NULL or unreachable pointer of a shard the plan copies);
 * UNSUPPORTED when the tables need more than RESHARD_STATIC_SCRATCH_BYTES (the message gives the
 * size; split the batch or use reshard_execute; checked before any CUDA call); CUDA. Calls no
 * cudaMalloc or cudaFree.
 */
#define RESHARD_STATIC_SCRATCH_BYTES (16u << 20)
int reshard_execute_static(const reshard_plan_t *plan, void *const *src_ptrs, void *const *dst_ptrs,
                           reshard_stream_t stream);

/* reshard_plan_stats -- fill *out (host only). */
int reshard_plan_stats(const reshard_plan_t *plan, reshard_stats_t *out);

/*
 * reshard_plan_regions -- copy up to `cap` planned regions into host arrays (introspection for
 * tests and tools). Per region i: tensor[i], src_rank[i] (pointer index of the chosen source),
 * dst_group[i] (plan-wide group id), and box lo/hi in global coordinates at
 * lo[i * RESHARD_MAX_DIMS + d], hi[...]. Any array may be NULL. *n_out gets the region count.
 */
int reshard_plan_regions(const reshard_plan_t *plan, int64_t cap, int32_t *tensor, int32_t *src_rank,
                         int32_t *dst_group, int64_t *lo, int64_t *hi, int64_t *n_out);

/*
 * reshard_plan_group_members -- destination pointer indices (within the tensor's run) of group
 * g. *n_out gets the member count; up to cap are written to members.
 */
int reshard_plan_group_members(const reshard_plan_t *plan, int64_t g, int64_t cap, int32_t *members,
                               int64_t *n_out);

/*
 * reshard_plan_items -- copy a device work-item table for inspection. set 0/1/2: the strided
 * copy items of the direct / pack / unpack pass; set 3/4/5: the transposing items of the same
 * passes (64 bytes each); set 6/7/8: the pair items of the same passes (96 bytes each).
 * Copy item: int64 src_off, dst_off, src_pitch, dst_pitch (elements); int32 rows, run (elements
 * per row), src (pointer-table index), group, esize (bytes), 3 x int32 padding. It moves `rows`
 * rows of `run` elements from src_off + r * src_pitch of pointer `src` to
 * member_offset + dst_off + r * dst_pitch of every member pointer of `group`.
 * Transposing item: int64 src_off, dst_off, src_pitch, dst_pitch; int32 rows, cols, src, group,
 * esize, slab, x, y. Element (r, c) moves from src_off + r * src_pitch + c to
 * member_offset + dst_off + c * dst_pitch + r; (x, y) are (c = 0, r = 0) in slab coordinates.
 * Pair item: int64 src_off[2], src_pitch[2], dst_off[2], dst_pitch[2]; int32 run[2], src[2],
 * rows, group, esize, kind. Row r of piece p is run[p] elements read at src_off[p] + r *
 * src_pitch[p] of pointer src[p] and written at member_offset + dst_off[p] + r * dst_pitch[p] of
 * every member of `group`. kind 0 (gather row; direct and unpack passes): one destination row of
 * two source pieces side by side (dst_off[1] = dst_off[0] + run[0]; in the unpack pass both pieces
 * are read from the receive buffer's entry). kind 1 (scatter row; pack pass): one source row into
 * two message blocks (src_off[1] = src_off[0] + run[0]). A pass's copy items that a pair item
 * covers carry 1 in their first padding word; the copy walkers skip them when pair items run,
 * and every other walk of the copy items (MXFP8, the allocation-free entry point) takes them.
 * Pointer table: [sources | destination data | destination scales | send buffer | receive
 * buffer] (pack items write the send buffer's group, unpack items read the receive buffer). Up to
 * cap items go to `items` (may be NULL); *n_out gets the count. Copy items are ordered largest
 * first (the walkers deal them round-robin to a persistent grid); transposing items are grouped
 * by element size (one launch per size).
 * Groups: group_start (n_groups + 2 entries incl. the workspace group), member_ptr and
 * member_off (elements) are copied when non-NULL; *n_groups_out / *n_members_out get sizes.
 */
int reshard_plan_items(const reshard_plan_t *plan, int set, int64_t cap, void *items, int64_t *n_out,
                       int32_t *group_start, int32_t *member_ptr, int64_t *member_off, int64_t *n_groups_out,
                       int64_t *n_members_out);

/*
 * reshard_plan_slabs -- the 2-D source slabs the transposing items read through TMA tensor maps
 * (encoded at execute time for the current pointers). Per slab, 6 int64 at out[6 i]: pointer-
 * table index, element size, element offset of (0, 0), columns (contiguous extent), rows, row
 * pitch (elements). Up to cap slabs are written; *n_out gets the count.
 */
int reshard_plan_slabs(const reshard_plan_t *plan, int64_t cap, int64_t *out, int64_t *n_out);

/*
 * reshard_plan_status -- the plan's device status word (0 = fine; bit 0: a TMA wait in the
 * transposing kernel gave up after its time limit and that launch's output is incomplete;
 * bit 1: the aligned walker met an item that was not 16-byte aligned for the launch's pointers
 * and skipped it, so that output is incomplete too).
 * Synchronizes the device, then reads the word; reset != 0 clears it. 0 before any execute.
 */
int reshard_plan_status(reshard_plan_t *plan, int32_t *status, int reset);

/* reshard_plan_destroy -- free the plan's host tables, device tables and workspace.
 * Safe on NULL. A plan that has executed first waits for the last execute it enqueued on each
 * stream (an event per stream, not a device-wide synchronize), so it is safe to destroy while its
 * work is in flight; it blocks until that work is done (cudaFree may also wait for the device).
 * Its waits and frees run in relaxed stream-capture mode, so a destroy (a garbage-collected
 * handle, say) does not invalidate a capture that another thread is recording. Executes captured
 * into a CUDA graph are not waited for: a plan must outlive every graph that captured its
 * executes, and the graph's launches must be complete before the plan is destroyed.
 * A plan that never executed frees host memory only. */
int reshard_plan_destroy(reshard_plan_t *plan);

/* reshard_last_error -- text of this thread's last error ("" if none). Valid until the next
 * call on the same thread. */
const char *reshard_last_error(void);

#ifdef __cplusplus
}
#endif
#endif /* RESHARD_H */
