/*
 * subm3d.h -- submanifold sparse 3D convolution (SubMConv3d: kernel 3, stride 1,
 * no padding) for NVIDIA B300 (sm_103a). C ABI of libsubm3d.so.
 *
 * What is computed (sources are the pages' titles and sections):
 *   "pixal3d_mrp_mlx README", scope table "Scope, measured against the shared
 *   core", and "pixal3d_mrp_mlx CLAUDE.md", "Measured facts": every SparseConv3d
 *   of the decoders is (c, out, 3) with stride 1 and no padding, which dispatches
 *   to the submanifold convolution; the README's introduction calls it the
 *   expensive part of the sparse decoders. Outputs exist only at the active input
 *   voxels:
 *
 *     out[i, o] = bias[o] + sum_{k : nbr[i,k] >= 0} sum_c W[o, kz, ky, kx, c] * feats[nbr[i,k], c]
 *
 *   with k = 9 (dz+1) + 3 (dy+1) + (dx+1) for the neighbour offset (dz, dy, dx) in
 *   {-1, 0, 1}^3 and (kz, ky, kx) = (dz+1, dy+1, dx+1) (cross-correlation, as a
 *   dense Conv3d). The weight layout [O, kz, ky, kx, I] with channels-last
 *   features is the one the README's commit header gives for the checkpoints.
 *
 * Beside the convolution, on the same voxel structures (same pages, same scope table,
 * which lists them next to SubMConv3d): a fused residual/activation epilogue
 * (subm3d_forward_ex), SparseDownsample(2) with its cache-paired SparseUpsample(2)
 * (subm3d_downsample, subm3d_upsample), and the sparse pixel-(un)shuffle on the same
 * subdivision (subm3d_spatial2channel, subm3d_channel2spatial).
 *
 * Conventions shared by every call:
 *   - All tensor pointers are DEVICE pointers owned by the caller. The library
 *     allocates no device memory; scratch space is the caller's `workspace`.
 *   - Arrays are dense row-major ("contiguous"); every pointer must be 16-byte
 *     aligned. Row strides are exactly the logical widths given.
 *   - `stream` is a cudaStream_t (NULL = the legacy default stream). Work is
 *     enqueued on it; subm3d_build_kmap additionally waits for it (see there).
 *   - Every call returns a subm3d_status. On failure, subm3d_last_error() gives a
 *     message (thread-local, valid until this thread's next call into the
 *     library) that names the argument and its value.
 *   - The calls use the current CUDA device. Host-side state that belongs to a device
 *     (kernel attributes, the device error word's address, the SM count) is looked up
 *     on the first call made with that device current and kept per device, so one
 *     process may use several devices (device ordinals below 64).
 */
#ifndef SUBM3D_H
#define SUBM3D_H

#include <stddef.h>
#include <stdint.h>
#include <cuda_runtime_api.h>

#if defined(__GNUC__)
#define SUBM3D_API __attribute__((visibility("default")))
#else
#define SUBM3D_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  SUBM3D_OK = 0,
  SUBM3D_ERR_ARG = -1,          /* a host-side argument check failed                    */
  SUBM3D_ERR_COORD_RANGE = -2,  /* a coordinate outside 0 <= z,y,x < res or 0 <= b <= 65534 */
  SUBM3D_ERR_DUPLICATE = -3,    /* two input rows share one (b, z, y, x)                */
  SUBM3D_ERR_HASH_FULL = -4,    /* a hash insert or lookup exceeded its probe limit     */
  SUBM3D_ERR_CUDA = -5,         /* a CUDA runtime call failed (message has the code)    */
  SUBM3D_ERR_UNSUPPORTED = -6,  /* valid but unsupported shape / dtype combination      */
  SUBM3D_ERR_WORKSPACE = -7,    /* workspace too small or misaligned                    */
  SUBM3D_ERR_DEVICE = -8        /* a kernel recorded an error: a bounded wait ran out,
                                   or nbr held an index outside [-1, N)                 */
} subm3d_status;

typedef enum { SUBM3D_F32 = 0, SUBM3D_BF16 = 1 } subm3d_dtype;

/* Pooling of subm3d_downsample. */
typedef enum {
  SUBM3D_POOL_MEAN = 0,  /* mean of the children present (fp32 sum / count)            */
  SUBM3D_POOL_MAX = 1    /* elementwise maximum of the children present                */
} subm3d_pool;

/* Activation of the fused epilogue (subm3d_forward_ex). */
typedef enum {
  SUBM3D_ACT_NONE = 0,  /* identity                                                  */
  SUBM3D_ACT_RELU = 1,  /* max(y, 0)                                                 */
  SUBM3D_ACT_SILU = 2   /* y * sigmoid(y) = y / (1 + exp(-y))                        */
} subm3d_act;

/* Largest accepted grid side and batch index. */
#define SUBM3D_MAX_RES 65535
#define SUBM3D_MAX_BATCH 65534

/*
 * Workspace bytes that subm3d_build_kmap needs for N voxels (the default hash table
 * is reserved for its worst case, one occupied block per voxel: the smallest power
 * of two >= 2N slots, at least 64, of 32 bytes each). Host-only, no CUDA
 * call. Returns 0 for N < 0.
 */
SUBM3D_API size_t subm3d_kmap_workspace_bytes(int64_t N);

/* Same, for an explicit hash capacity (a power of two >= 8; 0 = the default). */
SUBM3D_API size_t subm3d_kmap_workspace_bytes_ex(int64_t N, int64_t hash_capacity);

/*
 * Kernel map (neighbour table) of an active voxel set.
 *
 * The pages define the operation as submanifold (outputs only at active sites),
 * which needs, per active voxel, the index of each of its 27 neighbours; the map
 * is what the README's "spatial cache" lets several convolutions on one voxel set
 * share.
 *
 *   coords    device int32 [N, 4], rows (b, z, y, x); 0 <= b <= 65534, 0 <= z,y,x < res.
 *   N         number of active voxels, 0 <= N < 2^31. N = 0 is a no-op (OK).
 *   res       grid side, 1 <= res <= 65535.
 *   nbr       device int32 [N, 27], written: nbr[i, k] = index of the row of coords
 *             at coords[i] + offset k (same batch item), or -1 if that voxel is not
 *             active or lies outside [0, res)^3. Rows and values are in the caller's
 *             input order. Bit-exact (the answer is unique).
 *   workspace device scratch of at least subm3d_kmap_workspace_bytes(N) bytes,
 *             256-byte aligned; its contents on entry do not matter.
 *
 * Steps (all CUDA kernels on `stream`). A voxel's sort key is b above the interleaved
 * z/y/x bits (its Morton code); the low 6 bits of the code are its place inside its
 * aligned 4x4x4 block, the bits above name the block. Each voxel finds or claims its
 * block's slot in an open-addressing hash table (64-bit block key, 64-bit occupancy
 * mask, the block's first position; bounded linear probing) and sets its bit in the
 * mask (two voxels on one coordinate set one bit: fewer bits than voxels is a duplicate
 * coordinate). Only the occupied blocks' keys
 * are radix-sorted; a scan of their popcounts gives each block its first position, and
 * each voxel's position (first position + rank of its bit) puts the voxels in Morton
 * order. The 27 offsets of each voxel are probed by warps that take 32 consecutive
 * positions of that order and write each voxel's row of nbr contiguously.
 *
 * Synchronisation: the call waits for `stream` once, at its end, to read the
 * device status word, so it is not capturable into a CUDA graph. Errors found on
 * the device (COORD_RANGE, DUPLICATE, HASH_FULL) are returned by this same call;
 * nbr is then unspecified.
 */
SUBM3D_API int subm3d_build_kmap(const int32_t* coords, int64_t N, int32_t res, int32_t* nbr,
                      void* workspace, size_t ws_bytes, cudaStream_t stream);

/*
 * subm3d_build_kmap with two extras:
 *   order          device int32 [N] or NULL. If given, receives the Morton order:
 *                  order[s] = the input row at position s of the (b, Morton code)
 *                  ascending sort (stable, so ties keep input order).
 *   hash_capacity  0 for the default: a table of the smallest power of two >= N/4
 *                  slots (at least 64), rebuilt on the device at the workspace's full
 *                  size (the smallest power of two >= 2N, the worst case of one block
 *                  per voxel) when a block needs more than 32 probes; else a fixed
 *                  power of two >= 8 (slots, one per occupied block). A capacity below
 *                  the number of occupied blocks makes the call fail with
 *                  SUBM3D_ERR_HASH_FULL.
 */
SUBM3D_API int subm3d_build_kmap_ex(const int32_t* coords, int64_t N, int32_t res, int32_t* nbr,
                         int32_t* order, int64_t hash_capacity, void* workspace,
                         size_t ws_bytes, cudaStream_t stream);

/*
 * subm3d_build_kmap without the wait: every step is enqueued on `stream` and the call
 * returns at once, so a kernel-map build and the convolutions that use it can run back
 * to back on the GPU (or be captured together into a CUDA graph). Errors found on the
 * device (a coordinate out of range, a duplicate, a full hash table) are not returned
 * here: they are folded into the device error word, and the next
 * subm3d_forward_status() returns SUBM3D_ERR_COORD_RANGE, SUBM3D_ERR_DUPLICATE or
 * SUBM3D_ERR_HASH_FULL. nbr is then unspecified, but every entry the forward kernels
 * read is checked against [-1, N), so a forward on it never reads outside feats.
 * Host-side argument errors are returned as by subm3d_build_kmap.
 */
SUBM3D_API int subm3d_build_kmap_async(const int32_t* coords, int64_t N, int32_t res,
                                       int32_t* nbr, void* workspace, size_t ws_bytes,
                                       cudaStream_t stream);

/*
 * Occupancy-grouped tiles ("tile plan"). The hot-path forward works on tiles of 128
 * output rows and runs, for every tile, each of the 27 offsets at which any of its
 * rows has a neighbour. In input (or Morton) order nearly every tile has a neighbour
 * at nearly every offset, though on surfaces only about 11 of a voxel's 27 are there.
 * A tile plan orders the rows so that a tile's rows share their neighbour offsets:
 * within consecutive windows of the Morton order, voxels are sorted by their 27-bit
 * neighbour mask (bit k set when nbr[i, k] >= 0), Morton order kept among equal masks.
 * The forward then skips, per tile, every offset no row of the tile has (on the shell
 * workloads it runs 0.43-0.55 of the offsets instead of all of them), and stores each
 * output row through the plan's permutation, so `out` keeps the caller's input order.
 * The result is the same convolution (the formula at the top of this file).
 *
 * Plan layout (device buffer of subm3d_plan_bytes(N) bytes, 256-byte aligned, owned by
 * the caller; offsets from its start, each rounded up to 256 bytes):
 *   perm       int32 [N]           at 0: perm[r] = input row at plan row r
 *   nbr        int32 [N, 27]       next: row r = the neighbour-table row of input row
 *                                  perm[r] (values are input rows, as in subm3d_build_kmap)
 *   tile_mask  uint32 [ceil(N/128)] next: bit k of tile t set when some plan row in
 *                                  [128 t, 128 t + 128) has a neighbour at offset k
 * The window (voxels of the Morton order grouped together) trades the share of offsets
 * skipped against the spread of the rows a tile gathers; SUBM3D_GROUP_WINDOW is the
 * default. Window 1 is the Morton order itself (SUBM3D_GROUP_MORTON): its build needs
 * neither the grouping sort nor a second pass over the rows (the probe writes them in
 * plan order), its tiles skip the offsets none of their 128 spatially close voxels has
 * (about a sixth of them on shells), and it is the fastest plan end to end on the shell
 * workloads. The forward loads rows per thread on plans of windows below 4096 (whose
 * tiles keep most offsets) and copies whole rows through shared memory on sparser ones;
 * the choice is noted per plan buffer when it is built and changes no result.
 */
#define SUBM3D_GROUP_WINDOW 262144
#define SUBM3D_GROUP_MORTON 1   /* window 1: tiles of the Morton order */
#define SUBM3D_KMAP_ASYNC 1u   /* flags: return without waiting (see subm3d_build_kmap_async) */
SUBM3D_API size_t subm3d_plan_bytes(int64_t N);
/* Workspace bytes subm3d_build_kmap_grouped needs for N voxels (0 for N outside [0, 2^31)). */
SUBM3D_API size_t subm3d_kmap_grouped_workspace_bytes(int64_t N);

/*
 * Kernel map as a tile plan: the steps of subm3d_build_kmap up to the block table, then
 * each voxel's neighbour mask (a warp-cooperative pass over the Morton order), a stable
 * radix sort of the sorted positions by (window, mask), the plan's perm and tile masks,
 * and the neighbour rows written in plan order.
 *   coords, N, res  as subm3d_build_kmap.
 *   window          0 for SUBM3D_GROUP_WINDOW, else a power of two in [1, 2^30].
 *   plan            device buffer of at least subm3d_plan_bytes(N) bytes, written.
 *   workspace       device scratch of subm3d_kmap_grouped_workspace_bytes(N) bytes,
 *                   256-byte aligned.
 *   flags           0: wait for `stream` and return device-side errors as
 *                   subm3d_build_kmap does; SUBM3D_KMAP_ASYNC: do not wait (errors as
 *                   subm3d_build_kmap_async).
 * Bit-exact: the plan is a function of the voxel set and the window (stable sorts).
 */
SUBM3D_API int subm3d_build_kmap_grouped(const int32_t* coords, int64_t N, int32_t res,
                                         int64_t window, void* plan, size_t plan_bytes,
                                         void* workspace, size_t ws_bytes, unsigned flags,
                                         cudaStream_t stream);

/*
 * subm3d_forward_ex on a tile plan instead of an input-order nbr: feats, weight, bias,
 * residual, act, out, N, I, O, dtype and the kernels chosen are as there (feats,
 * residual and out in the caller's input order); `plan` is what
 * subm3d_build_kmap_grouped wrote for these N voxels. Asynchronous; a plan row whose
 * perm entry lies outside [0, N) is skipped and reported by subm3d_forward_status.
 */
SUBM3D_API int subm3d_forward_grouped(const void* feats, const void* plan, const void* weight,
                                      const void* bias, const void* residual, subm3d_act act,
                                      void* out, int64_t N, int32_t I, int32_t O,
                                      subm3d_dtype dtype, cudaStream_t stream);

/*
 * Kernel map without any device allocation. The pages have no counterpart to this
 * call; it exists for callers that cannot allocate device memory themselves -- a host
 * application that owns all device memory through its own pool and hands a plugin
 * only its input and output buffers, or a latency-critical loop where an allocation,
 * which may synchronise the device, is not acceptable.
 *
 * Same result and errors as subm3d_build_kmap (coords, N, res, nbr and stream as
 * there), but the scratch space (hash table, sort buffers, status word) is a 16 MiB
 * array compiled into the library, so N is limited to SUBM3D_NOALLOC_MAX_VOXELS; a
 * larger N returns SUBM3D_ERR_ARG before any device work. Every GPU that loads the
 * library keeps that array until the process exits. The first call on a device looks
 * up the array's device address. Like subm3d_build_kmap, the call waits for `stream`
 * at its end (it reads the build's status back), so no call can be captured into a CUDA
 * graph, and calls from one host thread never overlap on the GPU. All calls share the one array: each
 * call re-initialises what it reads, but calls made at the same time from several
 * host threads race on it.
 */
#define SUBM3D_NOALLOC_MAX_VOXELS 131072
SUBM3D_API int subm3d_build_kmap_noalloc(const int32_t* coords, int64_t N, int32_t res,
                                         int32_t* nbr, cudaStream_t stream);

/*
 * Forward pass of the submanifold convolution (the formula at the top of this file).
 *
 *   feats   device [N, I] of `dtype`, channels-last.
 *   nbr     device int32 [N, 27] as written by subm3d_build_kmap. An entry outside
 *           [-1, N) is treated as absent and recorded as SUBM3D_ERR_DEVICE (see
 *           subm3d_forward_status); it is never dereferenced.
 *   weight  device [O, 3, 3, 3, I] of `dtype` (the checkpoints' [O, kz, ky, kx, I]).
 *   bias    device [O] of `dtype`, or NULL for no bias.
 *   out     device [N, O] of `dtype`, written once per row (no atomics, no
 *           read-modify-write). Must not overlap the inputs.
 *   dtype   SUBM3D_BF16: bf16 inputs, fp32 accumulation (tcgen05 tensor cores,
 *           accumulator in tensor memory), bias added in fp32, output rounded to
 *           bf16 (nearest-even). Needs I % 8 == 0 and O % 8 == 0. I and O in
 *           {16, 32, 48, 64} run the narrow kernel (the gathered rows in tensor
 *           memory); other O <= 256 the kernel that stages them in shared memory
 *           (the rows copied there by tensor-copy gathers, four rows per copy, when
 *           I % 64 == 0, else by cp.async); larger O the CUDA-core kernel. All three compute
 *           the same sums (fp32 accumulation order may differ between them).
 *           SUBM3D_F32: fp32 inputs and accumulation on the CUDA cores.
 *   N, I, O N >= 0 (0 is a no-op), 1 <= I, O <= 4096.
 *
 * Fully asynchronous: only host-side argument checks are reported by the return
 * value. Device-side conditions are reported by subm3d_forward_status().
 */
SUBM3D_API int subm3d_forward(const void* feats, const int32_t* nbr, const void* weight,
                   const void* bias, void* out, int64_t N, int32_t I, int32_t O,
                   subm3d_dtype dtype, cudaStream_t stream);

/*
 * Forward pass with a fused block epilogue: the convolution above, then a residual
 * add and an activation, in the same kernel and the same single store per row:
 *
 *   out[i, o] = act( bias[o] + residual[i, o]
 *                    + sum_k sum_c weight[o, kz, ky, kx, c] * feats[nbr[i, k], c] )
 *
 * This is the tail of a residual block built on this convolution (the "pixal3d_mrp_mlx"
 * page, section "Scope, measured against the shared core", lists ResBlock-style and
 * ConvNeXt-style sparse blocks and activations next to SubMConv3d; the block
 * internals are not given there, so the epilogue offers the two pieces every such
 * block ends with). Several convolutions at one resolution share one nbr: build it
 * once, pass it to each call.
 *
 *   residual  device [N, O] of `dtype`, or NULL for none; 16-byte aligned. It may be
 *             the same buffer as `out` (an in-place residual block: each element is
 *             read before it is overwritten, by the same thread); any other overlap
 *             with `out`, and any overlap of `out` with feats, is not allowed.
 *   act       SUBM3D_ACT_NONE, SUBM3D_ACT_RELU or SUBM3D_ACT_SILU, applied in fp32 to
 *             the fp32 sum before the output is rounded to `dtype`.
 *
 * Other arguments, kernels, errors and asynchrony as subm3d_forward, which is this
 * call with residual = NULL and act = SUBM3D_ACT_NONE.
 */
SUBM3D_API int subm3d_forward_ex(const void* feats, const int32_t* nbr, const void* weight,
                                 const void* bias, const void* residual, subm3d_act act,
                                 void* out, int64_t N, int32_t I, int32_t O,
                                 subm3d_dtype dtype, cudaStream_t stream);

/*
 * SparseDownsample(2) and the subdivision its paired upsample needs. The
 * "pixal3d_mrp_mlx README" scope table lists SparseDownsample(2) (with a pooling mode,
 * per its status notes) and SparseUpsample(2) as the cache-paired inverse that reuses
 * the subdivision stored by the matching downsample; the pages give no more detail,
 * so this is the plain reading:
 *
 *   parent voxel of (b, z, y, x)  = (b, z >> 1, y >> 1, x >> 1)
 *   coarse voxels                 = the distinct parents, in (batch, Morton code) order
 *                                   (Morton: bit t of x -> 3t, of y -> 3t+1, of z -> 3t+2)
 *   coarse_feats[p, :]            = mean or max of feats over the children of p
 *   parent[i]                     = coarse row of fine row i
 *   child_mask[p]                 = OR over children of 1 << ((z&1)<<2 | (y&1)<<1 | (x&1))
 *
 * Steps: validate + pack and the kernel map's Morton radix sort (children of one
 * parent end up adjacent, since a parent's key is its children's key >> 3); parent
 * starts counted per 2048-position tile and scanned; one pass writes parent, coarse
 * coordinates, child masks and each parent's first sorted position; the pooling runs
 * a thread per (parent, 16 bytes of channels) in fp32, rounded once to the dtype.
 *
 *   coords        device int32 [N, 4] (b, z, y, x): as subm3d_build_kmap (range, no
 *                 duplicates; res as there). The coarse grid has side (res + 1) / 2.
 *   feats         device [N, C] of `dtype`, or NULL for the structure alone.
 *   mode          SUBM3D_POOL_MEAN or SUBM3D_POOL_MAX.
 *   coarse_coords device int32 [N, 4] (room for N rows; the first M are written).
 *   coarse_feats  device [N, C] of `dtype` (first M rows written); ignored if feats is NULL.
 *   parent        device int32 [N].
 *   child_mask    device uint8 [N] (first M written).
 *   M_out         HOST int64: the number of coarse voxels M (0 on failure).
 *   workspace     device scratch of subm3d_downsample_workspace_bytes(N), 256-byte
 *                 aligned; other pointers 16-byte aligned.
 *
 * Synchronises `stream` once (to read M and the status word), like subm3d_build_kmap;
 * the pooling kernel is enqueued before that wait and reads M on the device. Errors: ERR_ARG, ERR_WORKSPACE,
 * ERR_COORD_RANGE, ERR_DUPLICATE (outputs unspecified), ERR_CUDA, ERR_DEVICE.
 */
SUBM3D_API size_t subm3d_downsample_workspace_bytes(int64_t N);
SUBM3D_API int subm3d_downsample(const int32_t* coords, int64_t N, int32_t res, const void* feats,
                                 int32_t C, subm3d_dtype dtype, subm3d_pool mode,
                                 int32_t* coarse_coords, void* coarse_feats, int32_t* parent,
                                 uint8_t* child_mask, int64_t* M_out, void* workspace,
                                 size_t ws_bytes, cudaStream_t stream);

/*
 * subm3d_downsample on coordinates whose Morton order the caller already has: `order`
 * is what subm3d_build_kmap_ex wrote for the same coords and res (order[s] = input row
 * at position s of the (batch, Morton code) sort), device int32 [N], 16-byte aligned.
 * The radix sort is skipped: the sort keys are gathered in that order, and checked (rows
 * in [0, N), coordinates in the grid, keys ascending; SUBM3D_ERR_ARG otherwise). The
 * other arguments, the results and the one synchronisation are those of
 * subm3d_downsample.
 */
SUBM3D_API int subm3d_downsample_sorted(const int32_t* coords, int64_t N, int32_t res,
                                        const int32_t* order, const void* feats, int32_t C,
                                        subm3d_dtype dtype, subm3d_pool mode,
                                        int32_t* coarse_coords, void* coarse_feats,
                                        int32_t* parent, uint8_t* child_mask, int64_t* M_out,
                                        void* workspace, size_t ws_bytes, cudaStream_t stream);

/*
 * subm3d_downsample (order NULL) or subm3d_downsample_sorted (order given) without the
 * wait: every step is enqueued on `stream`, and M is written to the device word `M`
 * (int64, 8-byte aligned) instead of returned, so the call can be captured into a CUDA
 * graph and runs back to back with what follows. The outputs are sized for the worst
 * case M = N by the caller (coarse_coords [N, 4], coarse_feats [N, C], child_mask [N]);
 * rows [M, N) are left as they were. Errors found on the device (a coordinate outside the
 * grid, a duplicate, an order that is not the coordinates' Morton order) set *M to 0 and
 * are reported by the next subm3d_forward_status (SUBM3D_ERR_COORD_RANGE,
 * SUBM3D_ERR_DUPLICATE, SUBM3D_ERR_ARG). Host-side argument errors are returned here.
 */
SUBM3D_API int subm3d_downsample_async(const int32_t* coords, int64_t N, int32_t res,
                                       const int32_t* order, const void* feats, int32_t C,
                                       subm3d_dtype dtype, subm3d_pool mode,
                                       int32_t* coarse_coords, void* coarse_feats,
                                       int32_t* parent, uint8_t* child_mask, int64_t* M,
                                       void* workspace, size_t ws_bytes, cudaStream_t stream);

/*
 * SparseUpsample(2) with the subdivision a subm3d_downsample stored:
 *   fine_feats[i, :] = coarse_feats[parent[i], :]
 * (the fine voxel set is the one the downsample saw, in its row order).
 *
 *   coarse_feats  device [M, C] of `dtype`.
 *   parent        device int32 [N] from subm3d_downsample; an entry outside [0, M)
 *                 gives a zero row and is reported by subm3d_forward_status.
 *   fine_feats    device [N, C] of `dtype`; must not overlap coarse_feats.
 * All pointers 16-byte aligned. Fully asynchronous.
 */
SUBM3D_API int subm3d_upsample(const void* coarse_feats, int64_t M, int32_t C,
                               const int32_t* parent, int64_t N, subm3d_dtype dtype,
                               void* fine_feats, cudaStream_t stream);

/*
 * SparseSpatial2Channel(2), the sparse pixel-unshuffle paired with the same subdivision
 * (listed beside the down/upsample in the "pixal3d_mrp_mlx README" scope table; no
 * layout is given there). Reading: a parent's row holds its eight children's rows side by
 * side in child-bit order, zeros where a child is absent:
 *
 *   out[p, k*C .. k*C + C) = feats[i]  for the fine row i that is child k of p,
 *                            0         for k not in child_mask[p],
 *   k = (z&1)<<2 | (y&1)<<1 | (x&1) of coords[i].
 *
 *   feats       device [N, C] of `dtype`; coords device int32 [N, 4] (b, z, y, x), the
 *               fine voxels; parent device int32 [N] and child_mask device uint8 [M] from
 *               subm3d_downsample on the same coords.
 *   out         device [M, 8 C] of `dtype`.
 * A parent entry outside [0, M) is skipped and reported by subm3d_forward_status. All
 * pointers but child_mask 16-byte aligned. Fully asynchronous.
 */
SUBM3D_API int subm3d_spatial2channel(const void* feats, const int32_t* coords,
                                      const int32_t* parent, const uint8_t* child_mask, int64_t N,
                                      int64_t M, int32_t C, subm3d_dtype dtype, void* out,
                                      cudaStream_t stream);

/*
 * The inverse on the stored subdivision (channel2spatial):
 *   fine_feats[i, :] = coarse_feats[parent[i], k*C .. k*C + C),  k the child bit of coords[i].
 * coarse_feats device [M, 8 C]; fine_feats device [N, C]; a parent outside [0, M) gives a
 * zero row and is reported by subm3d_forward_status. 16-byte aligned; asynchronous.
 */
SUBM3D_API int subm3d_channel2spatial(const void* coarse_feats, const int32_t* coords,
                                      const int32_t* parent, int64_t N, int64_t M, int32_t C,
                                      subm3d_dtype dtype, void* fine_feats, cudaStream_t stream);

/*
 * Waits for `stream`, then reads and clears the device error word of the current
 * device, which the forward, upsample and pixel-shuffle kernels and the asynchronous
 * kernel-map builds report into. Returns SUBM3D_OK; SUBM3D_ERR_COORD_RANGE,
 * SUBM3D_ERR_DUPLICATE or SUBM3D_ERR_HASH_FULL when an asynchronous build found that;
 * else SUBM3D_ERR_DEVICE (the message says which condition: an nbr entry outside
 * [-1, N), a bounded pipeline wait that ran out, a parent entry outside [0, M), a plan
 * row naming no input row, an internal index error of a build). The word is shared by
 * all streams of the process.
 */
SUBM3D_API int subm3d_forward_status(cudaStream_t stream);

/*
 * Stage timing of the kernel-map builds, for measurement. While enabled (per host
 * thread; off by default), every kernel-map build made by this thread records a CUDA
 * event on its stream before its first stage and after each stage (block insert,
 * block compact, each block-sort pass, block starts, voxel scatter, probe; for the tile
 * plan the probe in Morton order with the masks, each grouping-sort pass and the plan
 * index). No extra synchronisation is added.
 * subm3d_kmap_stage_times waits for the last build's events and writes, for up to `max`
 * stages in order, the GPU milliseconds of each (ms[i]) and its name (names[i], a
 * static string); it returns the number of stages written, or a negative status.
 */
SUBM3D_API void subm3d_kmap_stage_timing(int enable);
SUBM3D_API int subm3d_kmap_stage_times(float* ms, const char** names, int max);

/* Thread-local message describing the last failure of this thread ("" if none). */
SUBM3D_API const char* subm3d_last_error(void);

/* Number of CUDA kernels this library has launched in this process (host counter). */
SUBM3D_API int64_t subm3d_kernel_launches(void);

#ifdef __cplusplus
}
#endif

#endif /* SUBM3D_H */
