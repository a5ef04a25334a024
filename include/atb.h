/*
 * atb.h -- C ABI of libatb, tiled tensor movement between HBM and shared
 * memory through the Tensor Memory Accelerator (TMA), for sm_103a (GB300).
 *
 * Sources the operations follow (web pages on the TMA):
 *   [L04]  "lesson 04: TMA - the async bulk copy engine"
 *   [ARC]  "GPU TMA tensor memory accelerator"
 *   [D76]  "Day 76: The Tensor Memory Accelerator (TMA)"
 *   [CDSL] "Understanding TMA loads in CuTe DSL"
 *
 * Conventions shared by every call
 *   - Coordinates, extents and box sizes are listed innermost (contiguous)
 *     dimension first: x, then y, ... ([D76] "Pitfalls", coordinates in the
 *     wrong order).  Coordinates are element offsets (int32) of a box's first
 *     element and may be negative or past the end: a load reads zero bytes
 *     there, a store drops those elements.
 *   - Listed origins may be any int32 within +-2^30 (a box beyond that is
 *     refused per box with ATB_ERR_COORD_RANGE in the device status).  The
 *     tensor-map engine can start a copy along the innermost dimension only
 *     on a 16-byte boundary (x * element_size a multiple of 16).  A listed box
 *     whose origin is off that grid is loaded through the map's second,
 *     one-chunk-wider descriptor (map_wide) from the origin rounded down to
 *     the grid, and the kernel's consumer threads cut the box out of that
 *     wider image (or, without map_wide, load it with plain loads); boxes
 *     written to a tensor from such an origin leave through aligned plain
 *     stores of 1, 2 or 4 bytes, each wholly inside the box.  The result is
 *     the same as for any other origin.  Tile-grid origins are always on the
 *     grid.
 *   - A "packed" buffer holds n box images back to back, image i at byte
 *     offset i * box_bytes, each byte-for-byte the shared-memory image of that
 *     box as the engine writes it (swizzle applied, stage base aligned to the
 *     swizzle period).  It must be 16-byte aligned.
 *   - Device pointers are plain CUDA device addresses owned by the caller.
 *     The library allocates device memory only once per device, lazily, for a
 *     small status block (see atb_device_status); call atb_init_device() before
 *     capturing any of these calls into a CUDA graph.
 *   - All launches are asynchronous on the caller's stream (NULL = the legacy
 *     default stream).  Host-detectable errors return before anything is
 *     launched; atb_last_error() then holds a sentence naming the rule, the
 *     dimension and the value.
 *   - atb_tile_load, atb_tile_store, atb_tile_roundtrip and
 *     atb_tile_roundtrip_add_f32 can be captured into CUDA graphs (stream
 *     capture) once atb_init_device() and one call of the same kind have run
 *     outside the capture on that device; a replay moves whatever the
 *     captured maps' buffers hold at replay time.
 *   - Pipeline kernels are launched with programmatic dependent launch: a
 *     launch may be scheduled while the previous kernel on the stream drains,
 *     sets up its shared memory, and waits for that kernel to complete (with
 *     its memory visible) before it touches global memory.  Stream order is
 *     therefore kept exactly; atb_launch.no_pdl = 1 turns the overlap off.
 *   - Errors raised inside a kernel (a wait that ran out of time, a listed
 *     origin beyond +-2^30) are recorded in the device status block and
 *     reported by atb_device_status(); the kernel returns early instead of
 *     hanging.
 *   - Every call may be made from any host thread.  atb_last_error() is
 *     kept per thread: it describes the last failed call of the calling
 *     thread.  Host-resident round trips (atb_tile_roundtrip_host) share
 *     one pair of transfer streams per device: concurrent calls are enqueued
 *     one at a time and their copies run in that order.
 */
#ifndef ATB_H
#define ATB_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define ATB_VERSION 1
#define ATB_MAX_RANK 5

/* A CUDA stream handle; layout-compatible with cudaStream_t / CUstream. */
typedef struct CUstream_st* atb_stream_t;

typedef enum {
    ATB_OK = 0,
    ATB_ERR_RANK = 1,            /* rank outside 1..5 */
    ATB_ERR_BOX_DIM = 2,         /* a box extent is 0 or above 256 */
    ATB_ERR_STRIDE_ALIGN = 3,    /* a byte stride (dims 1..rank-1) is not a multiple of 16 */
    ATB_ERR_BASE_ALIGN = 4,      /* global base address not 16-byte aligned */
    ATB_ERR_SMEM_ALIGN = 5,      /* packed buffer not 16-byte aligned */
    ATB_ERR_SWIZZLE = 6,         /* unknown swizzle mode */
    ATB_ERR_SWIZZLE_SPAN = 7,    /* swizzled box: inner box bytes differ from the swizzle span */
    ATB_ERR_INNER_BYTES = 8,     /* inner box bytes not a multiple of 16 */
    ATB_ERR_DTYPE = 9,           /* unknown element type */
    ATB_ERR_DRIVER = 10,         /* the driver's encoder is unavailable or refused the map */
    ATB_ERR_UNSUPPORTED_DEVICE = 11, /* current device is not compute capability 10.3 */
    ATB_ERR_SMEM_BUDGET = 12,    /* stages x stage bytes exceed the per-block shared memory */
    ATB_ERR_ARG = 13,            /* a null pointer, zero extent, bad stride or mismatched maps */
    ATB_ERR_TIMEOUT = 14,        /* (device) an mbarrier wait ran out of time */
    ATB_ERR_CUDA = 15,           /* a CUDA runtime call failed */
    ATB_ERR_COORD_ALIGN = 16,    /* not raised any more: off-grid origins along x are moved by
                                    threads; the number stays reserved */
    ATB_ERR_COORD_RANGE = 17,    /* (device) a box origin is beyond +-2^30 */
    ATB_ERR_STRIDE_RANGE = 18,   /* a byte stride (dims 1..rank-1) is 0 or not below 2^40 */
    ATB_ERR_DIM_RANGE = 19,      /* an extent is 0 or above 2^32 */
    ATB_ERR_RING_CHECK = 20      /* (device, checked launches) a ring stage held another box than
                                    the one the waiting role expected */
} atb_status;

typedef enum {
    ATB_U8 = 0, ATB_U16 = 1, ATB_U32 = 2, ATB_I32 = 3, ATB_U64 = 4, ATB_I64 = 5,
    ATB_F16 = 6, ATB_F32 = 7, ATB_F64 = 8, ATB_BF16 = 9
} atb_dtype;

typedef enum {
    ATB_SWIZZLE_NONE = 0, ATB_SWIZZLE_32B = 1, ATB_SWIZZLE_64B = 2, ATB_SWIZZLE_128B = 3
} atb_swizzle;

typedef enum {
    ATB_L2_PROMO_NONE = 0, ATB_L2_PROMO_64B = 1, ATB_L2_PROMO_128B = 2, ATB_L2_PROMO_256B = 3
} atb_l2_promotion;

/*
 * What a load puts in the image for elements outside the tensor ([ARC] "The
 * architecture: every piece explained": the descriptor carries the boundary
 * handling).  Stores never write outside the tensor, whatever the fill.
 */
typedef enum {
    ATB_OOB_ZERO = 0,            /* out-of-bounds load elements read as zero bytes */
    ATB_OOB_NAN = 1              /* floating-point types only (f16, bf16, f32, f64): they read as
                                    a NaN of the element type, the driver's NaN-request-zero-FMA
                                    fill; the bit pattern is the hardware's */
} atb_oob_fill;

/*
 * An encoded tensor map plus the parameters it was built from.  `map` is the
 * driver's 128-byte CUtensorMap ([D76] "The address arithmetic moves into a
 * descriptor": 128 opaque bytes); the rest is kept for validation, launch
 * sizing and the ragged-store path.  Treat it as read-only; it may be copied
 * by value, and must outlive the calls that use it (the kernels receive a copy
 * by value, so it may be freed once the call has returned).
 */
typedef struct {
    unsigned char map[128];
    unsigned char map_wide[128];      /* the same tensor with box[0] one 16-byte chunk wider and no
                                         swizzle: listed boxes whose x origin is off the 16-byte grid
                                         are loaded through it from the origin rounded down to the
                                         grid (see "Conventions") */
    uint64_t base;                    /* global address the map was encoded over */
    uint64_t dims[ATB_MAX_RANK];      /* innermost first */
    uint64_t strides[ATB_MAX_RANK];   /* byte strides; strides[0] = element size */
    uint32_t box[ATB_MAX_RANK];       /* innermost first */
    uint32_t elem_strides[ATB_MAX_RANK]; /* traversal step per dimension; [0] = 1 */
    uint32_t rank;
    uint32_t esize;                   /* element size in bytes */
    uint32_t dtype;                   /* atb_dtype */
    uint32_t swizzle;                 /* atb_swizzle */
    uint32_t l2_promotion;            /* atb_l2_promotion */
    uint32_t oob_fill;                /* atb_oob_fill */
    uint32_t box_bytes;               /* element size x product over d of ceil(box[d] / elem_strides[d]) */
    uint32_t wide_box0;               /* box[0] of map_wide (box[0] + 16 / element size), or 0 when
                                         there is none (box[0] would exceed 256, or the driver
                                         refused it): off-grid boxes are then loaded by threads */
    uint32_t magic;                   /* set by atb_encode_tiled */
} atb_tensor_map;

/* Pipeline shape of one launch.  Zero fields take the library defaults. */
typedef struct {
    uint32_t stages;       /* shared-memory ring depth, 1..16 (0 = the library's choice: 3, or
                              fewer if 3 do not fit, but for the consumers' own rings,
                              see atb_launch.consumer and atb_launch.release) */
    uint32_t ctas;         /* total CTAs; 0 = persistent grid of ctas_per_sm per SM */
    uint32_t ctas_per_sm;  /* 0 = the library's choice: about 96 KiB of stages per SM (1..8),
                              within what fits, but for the consumers' own rings (one or
                              two per SM) */
    uint32_t schedule;     /* 0 = box t goes to CTA t mod G; 1 = CTA b takes a contiguous run */
    uint32_t store_groups; /* bulk-store groups allowed in flight at once, 1..8, clamped to
                              `stages` (0 = the library's choice: 2, but for the consumers'
                              own rings); a stage is recycled as soon as the group that
                              stores from it has finished reading it.  Giving any of
                              stages, ctas_per_sm or store_groups turns the own rings off:
                              the other two then take the common defaults */
    uint32_t l2_hints;     /* ATB_HINT_* bits: L2 eviction policy of the box loads and stores */
    uint32_t no_pdl;       /* 1 = launch without programmatic dependent launch (see below) */
    uint32_t poll_suspend_ns; /* mbarrier waits: suspend-time hint per poll in ns (0 = hardware default) */
    uint32_t prefetch_boxes;  /* tensor loads: prefetch the box this many boxes ahead into L2 with
                                 cp.async.bulk.prefetch.tensor (0 = off) */
    uint32_t checks;          /* ATB_CHECK_* bits: consistency checks inside the kernel (0 = none) */
    uint32_t consumer;        /* tile-grid launches: ATB_CONSUMER_* (0 = the library's choice) */
    uint32_t release;         /* the drain's stage release: ATB_RELEASE_* (0 = the library's choice) */
} atb_launch;

/*
 * atb_launch.consumer, for launches over the tile grid whose every box leaves
 * through one engine copy (gathers; stores and round trips whose destination
 * holds the whole grid and whose rows end on 16-byte boundaries).  Other
 * launches ignore it, and launches with prefetch_boxes or poll_suspend_ns set
 * always take the warp consumer.
 *   ATB_CONSUMER_AUTO   the library's choice: the one-thread drain for
 *                       stages of 32 KiB and more, and for stages of 4 to
 *                       32 KiB when the launch leaves stages, store_groups
 *                       and ctas_per_sm at 0 (the drain then runs its own
 *                       ring: 64 KiB of stages per SM for boxes being loaded
 *                       or landed plus 48 KiB of store groups, one CTA per
 *                       SM, or below 8 KiB two CTAs with 32 + 16 KiB each;
 *                       each stage freed before the next store is issued);
 *                       the warp consumer otherwise (the faster choice for
 *                       each case on GB300)
 *   ATB_CONSUMER_DRAIN  one consumer thread per CTA waits for each stage and
 *                       issues its drain copy; fewest instructions per box
 *   ATB_CONSUMER_WARP   a consumer warp follows every box and its lane 0
 *                       issues the drain copy (the consumer that can also
 *                       write boxes with plain clipped stores)
 */
#define ATB_CONSUMER_AUTO  0u
#define ATB_CONSUMER_DRAIN 1u
#define ATB_CONSUMER_WARP  2u

/*
 * atb_launch.release: when a stage whose box is being stored is handed back
 * to the producer (every consumer).
 *   ATB_RELEASE_AUTO          the library's choice: before the next store on
 *                             the drain's own ring and on the several-warp
 *                             consumer's own ring (16-32 KiB stages, no shape
 *                             given: two CTAs per SM, 32 KiB of stages for
 *                             boxes being loaded or landed and 48 KiB of
 *                             store groups each), after it otherwise
 *   ATB_RELEASE_AFTER_STORE   after storing box k the consumer waits until at
 *                             most store_groups - 1 groups still read and
 *                             frees the stage of box k - store_groups + 1
 *   ATB_RELEASE_BEFORE_STORE  after box k lands the consumer waits until at
 *                             most store_groups - 1 groups still read and
 *                             frees the stage of box k - store_groups, then
 *                             stores box k: the load into the freed stage is
 *                             issued ahead of the store (the drain first
 *                             pauses for about 64 ns).  Needs store_groups <
 *                             stages (ATB_ERR_ARG otherwise).
 */
#define ATB_RELEASE_AUTO         0u
#define ATB_RELEASE_AFTER_STORE  1u
#define ATB_RELEASE_BEFORE_STORE 2u

/*
 * atb_launch.checks bits.
 *
 * ATB_CHECK_RING  stage bookkeeping check, a debugging aid for the ring (the
 *   pages' failure modes of a TMA pipeline are silent: a consumer that waits
 *   on the wrong phase parity reads a stale or half-written box, "Understanding
 *   TMA loads in CuTe DSL", "Issue the load and wait for its phase"; "Day 76:
 *   The Tensor Memory Accelerator (TMA)", "Pitfalls").  Each CTA keeps two
 *   shadow words per stage in shared memory.  Before arming a stage the
 *   producer writes the number of the box it is about to load there; after its
 *   full-barrier wait the consumer compares that number with the box it
 *   expects.  When a stage is released the consumer writes the number of the
 *   box it is done with; after its empty-barrier wait the producer compares it
 *   with the stage's previous box.  The barriers' release/acquire order makes
 *   each shadow write visible to the waiting role.  A mismatch records
 *   ATB_ERR_RING_CHECK (where = 6 producer, 7 consumer) and the launch goes
 *   on; no wait is added.  Costs a few shared-memory accesses per box.
 */
#define ATB_CHECK_RING 1u

/* atb_launch.l2_hints bits */
#define ATB_HINT_LOAD_EVICT_FIRST  1u
#define ATB_HINT_STORE_EVICT_FIRST 2u
#define ATB_HINT_STORE_EVICT_LAST  4u

/* Contents of the device status block (one per device). */
typedef struct {
    int32_t code;          /* atb_status of the first device-side error, 0 = none */
    int32_t block;         /* CTA that recorded it */
    int32_t tile;          /* box index (position in the list or grid) it was working on */
    int32_t where;         /* 1 producer wait, 2 consumer wait, 3 producer issue, 4 consumer issue,
                              5 self-test wait, 6 producer ring check, 7 consumer ring check */
    uint32_t errors;       /* number of device-side errors recorded since the last reset */
    uint32_t reserved[3];
} atb_device_report;

/* Library version (ATB_VERSION). */
int atb_version(void);

/* sizeof(atb_tensor_map), so bindings can check their mirror of the struct. */
size_t atb_tensor_map_size(void);

/* Human-readable name of a status code.  Static storage; never NULL. */
const char* atb_status_string(atb_status s);

/* The last host-side error of this thread, as a sentence ("" if none). */
const char* atb_last_error(void);

/*
 * atb_encode_tiled -- build and validate a tiled tensor map.
 *
 * [D76] "The address arithmetic moves into a descriptor" and "Pitfalls"
 * (the encoder returns a bare invalid-value error for any broken rule),
 * [L04] "The real toolchain - PTX and the descriptor object" (the map is
 * encoded once on the host and handed to the kernel as a grid constant),
 * [ARC] "The architecture: every piece explained" (shape, strides, box and
 * out-of-bounds fill live in the descriptor).
 *
 * Checks, each with its own status before the driver is asked:
 *   rank in 1..5                                 -> ATB_ERR_RANK
 *   dtype known                                  -> ATB_ERR_DTYPE
 *   gbase non-null and 16-byte aligned           -> ATB_ERR_ARG / ATB_ERR_BASE_ALIGN
 *   every dims[d] in 1..2^32                     -> ATB_ERR_DIM_RANGE
 *   strides_bytes[d] (d = 1..rank-1) multiple of 16 -> ATB_ERR_STRIDE_ALIGN
 *   strides_bytes[d] in 16..2^40-16               -> ATB_ERR_STRIDE_RANGE
 *   (strides need not grow with d: permuted views are passed as they are)
 *   every box[d] in 1..256                       -> ATB_ERR_BOX_DIM
 *   box[0] * element size multiple of 16         -> ATB_ERR_INNER_BYTES
 *   swizzle known                                -> ATB_ERR_SWIZZLE
 *   swizzled: box[0] * element size == span (32/64/128) -> ATB_ERR_SWIZZLE_SPAN
 *   elem_strides NULL, or [0] == 1 and each entry in 1..8 -> ATB_ERR_ARG
 *   l2_promotion known, oob_fill known           -> ATB_ERR_ARG
 *   oob_fill ATB_OOB_NAN with an integer dtype    -> ATB_ERR_DTYPE
 * then fetches cuTensorMapEncodeTiled through the runtime's driver entry point
 * (no libcuda link) and encodes; a driver refusal -> ATB_ERR_DRIVER.
 *
 *   out           caller-owned result (any alignment)
 *   gbase         device address of element (0, ..., 0)
 *   dims          rank extents, innermost first
 *   strides_bytes rank entries: strides_bytes[0] is ignored (the innermost
 *                 dimension is contiguous), strides_bytes[d] is the byte
 *                 distance between neighbours along dimension d; NULL is not
 *                 allowed for rank > 1
 *   box           rank box extents, innermost first
 *   elem_strides  NULL (all 1), or rank traversal steps: along dimension d
 *                 the box visits elements origin, origin + e, ... inside its
 *                 extent, ceil(box[d] / e) of them, packed densely in the
 *                 image (the driver's elementStrides).  The innermost step
 *                 must be 1 (the engine has no step along the contiguous
 *                 dimension).  The tile grid still advances by box[d].
 */
atb_status atb_encode_tiled(atb_tensor_map* out, atb_dtype dtype, uint32_t rank, void* gbase,
                            const uint64_t* dims, const uint64_t* strides_bytes,
                            const uint32_t* box, const uint32_t* elem_strides,
                            atb_swizzle swizzle, atb_l2_promotion l2_promotion,
                            atb_oob_fill oob_fill);

/* Bytes of one box image of a map (see atb_tensor_map.box_bytes); 0 if map is NULL. */
size_t atb_box_bytes(const atb_tensor_map* map);

/* Number of boxes that tile the whole tensor, edge boxes included; 0 if map is NULL. */
uint64_t atb_grid_tiles(const atb_tensor_map* map);

/*
 * Dynamic shared memory one CTA of a pipeline with `stages` stages over this
 * map needs (stage ring, barriers, alignment slack), in *bytes.
 * ATB_ERR_SMEM_BUDGET if it exceeds the device's per-block limit (the
 * requested value is still written).
 */
atb_status atb_pipeline_smem_bytes(const atb_tensor_map* map, uint32_t stages, size_t* bytes);

/*
 * The launch shape of this host thread's most recent tile load, store or round
 * trip call (the regular, host-buffer and allocation-free entry points alike):
 * what the library resolved from atb_launch and its defaults.  All fields are
 * 0 when that call launched nothing (no boxes, or refused).  Reading it
 * touches no device.
 *   consumer      ATB_CONSUMER_DRAIN or ATB_CONSUMER_WARP for tile-grid
 *                 launches; ATB_CONSUMER_WARPS for launches with several
 *                 consumer warps (coordinate lists and the fp32 update)
 *   release       ATB_RELEASE_AFTER_STORE or ATB_RELEASE_BEFORE_STORE
 *   stages, store_groups, ctas_per_sm, ctas (the grid), threads per CTA,
 *   smem_bytes (dynamic shared memory per CTA), boxes (boxes the launch moves)
 * ATB_ERR_ARG if out is NULL.
 */
#define ATB_CONSUMER_WARPS 3u
typedef struct {
    uint32_t consumer;
    uint32_t release;
    uint32_t stages;
    uint32_t store_groups;
    uint32_t ctas_per_sm;
    uint32_t ctas;
    uint32_t threads;
    uint32_t smem_bytes;
    uint32_t boxes;
    uint32_t reserved[3];
} atb_launch_shape;

atb_status atb_last_launch(atb_launch_shape* out);

/*
 * atb_tile_load -- gather boxes into a packed buffer of shared-memory images.
 *
 * [L04] "What the issuing thread actually does" and "Load completion - the
 * mbarrier and the byte budget"; [D76] "An exact round trip"; [CDSL] "Issue
 * the load and wait for its phase".  A persistent, warp-specialised CTA ring:
 * one producer thread arms stage s with arrive.expect_tx(box_bytes) and issues
 * one cp.async.bulk.tensor per box; one consumer thread waits on the stage's
 * phase and drains the landed image with a 1-D bulk store to
 * d_packed + i * box_bytes, recycling the stage after the bulk group's reads.
 * Calls with a coordinate list run four consumer warps: a listed box whose x
 * origin is off the 16-byte grid is loaded through map_wide from the origin
 * rounded down to the grid, and those warps cut its image out of the wider
 * one (without map_wide they build it with plain loads, writing the same
 * fill bytes as the engine outside the tensor) before it is drained.
 *
 *   src       encoded map of the source tensor
 *   d_coords  device array of n * rank int32 origins, innermost first; NULL =
 *             every box of the tile grid in row-major tile order (innermost
 *             tile index fastest), n is then ignored.  The producer thread
 *             reads each origin once and hands it to the consumers with the
 *             stage.
 *   d_packed  device output, 16-byte aligned, n * box_bytes bytes
 *   launch    NULL for defaults
 * n = 0 launches nothing.  The kernel reads d_coords and the source, and
 * writes d_packed, while it runs on `stream`: the caller keeps them allocated
 * and unchanged (d_packed unread) until the stream has passed the call.
 */
atb_status atb_tile_load(const atb_tensor_map* src, const int32_t* d_coords, uint64_t n,
                         void* d_packed, const atb_launch* launch, atb_stream_t stream);

/*
 * atb_tile_store -- write packed box images back into a tensor.
 *
 * [L04] "Store completion - commit group and wait group"; [D76] "Exercise",
 * "Hint 2" and "Solution" (the shared-to-global direction, completed through
 * a bulk async group, not an mbarrier).  The producer brings image i into a
 * stage with a 1-D bulk copy counted by the stage's mbarrier; the consumer
 * issues the tensor store, commits it and recycles the stage after
 * wait_group.read.  Elements outside the tensor are not written.  A box whose
 * origin is negative in any dimension is written by the consumer threads with
 * plain clipped stores instead (a tensor store may not start before the
 * tensor), and so is a box whose x origin is off the 16-byte grid, and a box
 * that crosses the end of a row whose byte length (dims[0] x element size) is
 * not a multiple of 16: the engine writes the last 16-byte chunk of such a
 * row whole, which would spill past the row.
 * Calls with a coordinate list run four consumer warps, which share those
 * clipped stores; calls over the tile grid run one.
 * Boxes that overlap with different contents land in an unspecified order.
 *
 *   dst       encoded map of the destination tensor
 *   d_coords  as for atb_tile_load (NULL = tile grid)
 *   d_packed  device input, 16-byte aligned, n * box_bytes bytes
 */
atb_status atb_tile_store(const atb_tensor_map* dst, const int32_t* d_coords, uint64_t n,
                          const void* d_packed, const atb_launch* launch, atb_stream_t stream);

/*
 * atb_tile_roundtrip -- move boxes from one tensor to another through shared
 * memory: load with the source map, store with the destination map.
 *
 * [D76] "Exercise" (a second map over the output; the only global traffic is
 * two bulk tensor instructions), [L04] "Why this only pays off inside a
 * pipeline" and [ARC] "The architecture" / "End-to-end flow" (an N-stage ring,
 * stage k mod N, a stage refilled only after its consumer is done).
 * Result = store(dst, coords, load(src, coords)).
 *
 *   src, dst  maps with equal rank, element size, box extents and swizzle
 *             (ATB_ERR_ARG otherwise); extents and strides may differ.
 *             Source and destination memory must not overlap.
 *   d_coords  as for atb_tile_load (NULL = the source's tile grid)
 */
atb_status atb_tile_roundtrip(const atb_tensor_map* src, const atb_tensor_map* dst,
                              const int32_t* d_coords, uint64_t n, const atb_launch* launch,
                              atb_stream_t stream);

/*
 * atb_tile_roundtrip_host -- the full-grid round trip for tensors that live
 * in host memory: copy the source host -> device, move every box through
 * shared memory into the destination, copy the destination device -> host.
 *
 * The tile grid is cut into `slabs` runs of whole box rows along the
 * outermost dimension.  Slab j's host-to-device copy, its boxes' round trip
 * and its device-to-host copy run on three streams ordered by events, so the
 * copies of one slab overlap the work of the others ([L04] "Why this only
 * pays off inside a pipeline", applied to whole slabs).  The call is ordered
 * after earlier work on `stream`, and later work on `stream` runs after it.
 *
 *   src, dst  maps over caller-owned DEVICE buffers (staging); equal rank and
 *             extents; box, element size and swizzle as for
 *             atb_tile_roundtrip
 *   h_src     host memory laid out exactly as `src` describes its device
 *             buffer (same byte offsets); pinned memory lets copies overlap
 *   h_dst     host memory laid out as `dst` describes its device buffer;
 *             bytes between rows (padding) may be overwritten with the
 *             device buffer's contents
 *   slabs     0 = 12; clamped to 1..64 and to the number of box rows.  When
 *             the outermost stride does not step over the whole inner span
 *             (a permuted view), the call uses one slab.
 * Not for concurrent use from several host threads on one device (the
 * per-device streams and events are shared; calls serialise their enqueue).
 */
atb_status atb_tile_roundtrip_host(const atb_tensor_map* src, const atb_tensor_map* dst,
                                   const void* h_src, void* h_dst, uint32_t slabs,
                                   const atb_launch* launch, atb_stream_t stream);

/*
 * atb_tile_roundtrip_add_f32 -- the round trip with an elementwise fp32 update
 * in shared memory: every element of each landed box becomes x + addend
 * (IEEE round-to-nearest, denormals kept) before the box is stored.
 *
 * [D76] "Exercise", "Hint 1", "Hint 2" and "Solution": the threads change
 * the tile in shared memory through the generic proxy, each writer then
 * publishes its writes with fence.proxy.async, the group meets at a barrier
 * and one thread issues the tensor store, completed through a bulk async
 * group.  Two consumer warps update each stage; one producer thread loads.
 *
 *   src, dst  ATB_F32 maps with equal rank, box extents and swizzle
 *             (ATB_ERR_DTYPE / ATB_ERR_ARG otherwise)
 *   d_coords  as for atb_tile_load (NULL = the source's tile grid)
 * Result = store(dst, coords, load(src, coords) + addend).  Elements outside
 * the source read as 0 and are therefore stored as 0 + addend where they lie
 * inside the destination.
 */
atb_status atb_tile_roundtrip_add_f32(const atb_tensor_map* src, const atb_tensor_map* dst,
                                      const int32_t* d_coords, uint64_t n, float addend,
                                      const atb_launch* launch, atb_stream_t stream);

/*
 * Allocate this device's status block now (it is otherwise allocated on the
 * first launch on the device).  Call before capturing launches in a graph.
 */
atb_status atb_init_device(void);

/*
 * After the work already queued on `stream`, copy the current device's
 * status block into *report (may be NULL) and reset it, then wait for that.
 * Returns the recorded code (ATB_OK if none).  The block is shared by every
 * stream of the device: kernels still running on other streams may record
 * errors after the read; synchronise them first to include them.
 */
atb_status atb_device_status(atb_stream_t stream, atb_device_report* report);

/*
 * Whether the current device's status block (see atb_init_device) has been
 * allocated in this process: 1 yes, 0 no, -1 if the current device cannot be
 * read.  Allocates nothing and launches nothing.
 */
int atb_status_block_allocated(void);

/* Limit for every mbarrier wait inside the kernels, in nanoseconds of the
 * GPU's global timer (default 1e9 = one second).  0 restores the default. */
void atb_set_wait_timeout_ns(uint64_t ns);

/*
 * Self-test of the bounded wait: one CTA waits on an mbarrier that nothing
 * will complete, gives up after timeout_ns, records ATB_ERR_TIMEOUT (where =
 * 5) in the status block and returns.  No copy is in flight.  Returns the
 * launch status; read the outcome with atb_device_status().
 */
atb_status atb_selftest_wait_timeout(uint64_t timeout_ns, atb_stream_t stream);

/*
 * atb_tile_roundtrip_noalloc -- atb_tile_roundtrip for callers that must not
 * allocate device memory.  The pages have no counterpart to this call.
 *
 * atb_tile_roundtrip records kernel errors in a status block that the library
 * obtains with cudaMalloc the first time it runs on a device.  Some callers
 * cannot let that happen: code being captured into a CUDA graph in global
 * capture mode (where cudaMalloc is refused), services that reserve all of a
 * GPU's memory for their own pool at start-up and forbid any later
 * allocation, and latency-critical threads that must not take the driver's
 * allocation path.  This entry point moves the same boxes with the same kernel
 * but keeps the error record in a static device array of
 * ATB_NOALLOC_SCRATCH_BYTES bytes that is part of the library image: every GPU
 * that loads the library holds those bytes until the process exits.  It calls
 * no cudaMalloc, cudaFree or allocating library routine.
 *
 *   src, dst, d_coords, n, launch, stream  as for atb_tile_roundtrip
 *   report  NULL: return right after the launch (kernel errors are then not
 *           reported).  Otherwise host memory: the call waits for `stream`,
 *           copies the error record there and returns its code.
 *
 * Scratch: this kernel needs sizeof(atb_device_report) bytes whatever the
 * problem size; a call that would need more than ATB_NOALLOC_SCRATCH_BYTES is
 * rejected with ATB_ERR_ARG before anything is launched.  Every call on a
 * device shares the one array, which keeps the last call's record; each call
 * clears it (an asynchronous memset on `stream`) before its launch.  Calls
 * whose work overlaps on the GPU (different streams, or a second call issued
 * before the first one's report was read) race on that record.
 * The first call on each device looks up the array's device address (one
 * runtime query, with that device current); make that first call before any
 * stream capture begins.
 */
#define ATB_NOALLOC_SCRATCH_BYTES 256
atb_status atb_tile_roundtrip_noalloc(const atb_tensor_map* src, const atb_tensor_map* dst,
                                      const int32_t* d_coords, uint64_t n, const atb_launch* launch,
                                      atb_stream_t stream, atb_device_report* report);

/*
 * Bandwidth ablations (flat copies of `bytes` bytes, both pointers 16-byte
 * aligned, bytes a multiple of 16):
 *   atb_copy_cpasync  thread-issued cp.async (LDGSTS, 16 B per lane) into a
 *                     shared-memory ring, then ld.shared.v4 / st.global.v4
 *                     ([L04] "What the issuing thread actually does": the
 *                     Ampere-style copy where every lane issues its slice);
 *   atb_copy_ldst_v4  plain coalesced ld.global.v4 / st.global.v4 through
 *                     registers ([D76] the per-thread loads of the diagram in
 *                     "The address arithmetic moves into a descriptor");
 *   atb_copy_memcpy   cudaMemcpyAsync device-to-device.
 * `launch` may be NULL; only `ctas`, `ctas_per_sm` and `stages` are used.
 */
atb_status atb_copy_cpasync(const void* d_src, void* d_dst, size_t bytes, const atb_launch* launch,
                            atb_stream_t stream);
atb_status atb_copy_ldst_v4(const void* d_src, void* d_dst, size_t bytes, const atb_launch* launch,
                            atb_stream_t stream);
atb_status atb_copy_memcpy(const void* d_src, void* d_dst, size_t bytes, atb_stream_t stream);

#ifdef __cplusplus
}
#endif

#endif /* ATB_H */
