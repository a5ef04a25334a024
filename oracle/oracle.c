/*
 * Plain CPU oracle for tiled tensor movement through a tensor-map descriptor.
 *
 * TEST INFRASTRUCTURE ONLY.  The test suite, the smoke check and the
 * benchmark's CPU-baseline leg are the only callers.  Nothing here is shared
 * with the CUDA library: no header, helper, table or constant.  Every function
 * is the definition written out, element by element and byte by byte, in the
 * order the pages describe it, with no blocking, fusion or reordering.
 *
 * Sources (web pages on the Tensor Memory Accelerator):
 *   [L04] "lesson 04: TMA - the async bulk copy engine"
 *   [ARC] "GPU TMA tensor memory accelerator"
 *   [D76] "Day 76: The Tensor Memory Accelerator (TMA)"
 *   [CDSL] "Understanding TMA loads in CuTe DSL"
 *
 * Readings taken where the pages are silent (each one is listed with the
 * design notes of the repository):
 *   R1  out-of-bounds elements of a load are all-zero bytes ([ARC] "The
 *       architecture: every piece explained": the engine can zero-fill; [L04]
 *       "The real toolchain" encodes FLOAT_OOB_FILL_NONE).
 *   R2  a store writes only in-bounds elements; the rest are dropped.
 *   R3  the box image is laid out row-major over the box, innermost dimension
 *       contiguous, and the swizzle permutes byte offsets of that image as
 *       CuTe's Swizzle<B,M,S> with M = 4 (16-byte chunks) and S = 3 (the chunk
 *       index is XORed with bits taken 3 positions higher, i.e. with the
 *       128-byte row index), B = 0/1/2/3 for none/32B/64B/128B.
 *   R4  the packed buffer holds box i at byte offset i*box_bytes, in the order
 *       of the coordinate list; the full tile grid is enumerated row-major over
 *       tile indices, innermost tile index fastest.
 *   R5  a traversal step e along an outer dimension makes the box visit every
 *       e-th element of its extent (ceil(box / e) elements), packed densely in
 *       the image; the tile grid still advances by the box extent.
 *   R6  with the NaN fill the descriptor can request instead of zeros, an
 *       out-of-bounds load element reads as some NaN of the element type; no
 *       page gives the bit pattern, so the oracle names the filled bytes
 *       (oracle_tile_oob_mask) rather than their values.
 *
 * Parity of every function is pinned by tests that do not re-type these
 * formulas: the byte counts and tile positions the pages print, brute-force
 * bijection and closed-form checks of the swizzle, an independent gather by
 * zero-padded array slicing on tiny tensors, and store-after-load identity.
 */
#include "oracle.h"

#include <stdlib.h>
#include <string.h>

/*
 * Swizzle<B,4,3> on a byte offset.  [CDSL] "Describe the memory layout first"
 * builds the shared tile as make_swizzle(0, 4, 3) composed with a row-major
 * layout and states that zero swizzle bits leave every offset unchanged.  With
 * B bits the mask selects offset bits [7, 7+B) and XORs them into bits
 * [4, 4+B): the 16-byte chunk number inside a 128-byte row is XORed with the
 * low B bits of the row number.  [L04] "The descriptor records the layout,
 * including the swizzle": the engine applies this as bytes land in shared
 * memory, with no separate pass.
 */
uint64_t oracle_swizzle(uint64_t offset, int32_t bits)
{
    const int32_t M = 4;  /* 16-byte chunks stay intact */
    const int32_t S = 3;  /* source bits sit S positions above the chunk bits */
    uint64_t low_bits = ((uint64_t)1 << bits) - 1;
    uint64_t source_mask = low_bits << (M + S);
    return offset ^ ((offset & source_mask) >> S);
}

/* Traversal step along dimension d (1 when unset).  Reading R5: a box with
 * step e along d visits elements origin, origin + e, ... inside its extent,
 * ceil(box / e) of them; the innermost dimension is always contiguous. */
static uint64_t step_along(const oracle_view* v, int32_t d)
{
    return v->estr[d] > 1 ? v->estr[d] : 1;
}

/* Elements the box visits along dimension d. */
static uint64_t visits_along(const oracle_view* v, int32_t d)
{
    return (v->box[d] + step_along(v, d) - 1) / step_along(v, d);
}

/* [D76] "The address arithmetic moves into a descriptor": a 64x64 float box
 * is a 16384-byte transfer; the box size is the product of its extents (of
 * the visited elements when a traversal step is set). */
uint64_t oracle_box_bytes(const oracle_view* v)
{
    uint64_t elems = 1;
    for (int32_t d = 0; d < v->rank; ++d) elems *= visits_along(v, d);
    return elems * (uint64_t)v->esize;
}

/* Number of boxes along dimension d when the tensor is cut into whole boxes,
 * the last one possibly hanging over the edge. */
static uint64_t tiles_along(const oracle_view* v, int32_t d)
{
    return (v->dims[d] + v->box[d] - 1) / v->box[d];
}

/* [CDSL] "The work assigned to each block": tile (b, j) of a row-major matrix
 * covers rows [64b, 64(b+1)) and columns [256j, 256(j+1)); in general the
 * tile with index t_d along dimension d starts at element t_d * box[d]. */
uint64_t oracle_grid_count(const oracle_view* v)
{
    uint64_t count = 1;
    for (int32_t d = 0; d < v->rank; ++d) count *= tiles_along(v, d);
    return count;
}

void oracle_grid_coords(const oracle_view* v, int32_t* coords)
{
    uint64_t count = oracle_grid_count(v);
    for (uint64_t t = 0; t < count; ++t) {
        uint64_t rest = t;
        for (int32_t d = 0; d < v->rank; ++d) {
            uint64_t n_d = tiles_along(v, d);
            uint64_t t_d = rest % n_d;
            rest /= n_d;
            coords[t * (uint64_t)v->rank + (uint64_t)d] = (int32_t)(t_d * v->box[d]);
        }
    }
}

/*
 * Box element with linear index e (innermost fastest) of the box whose origin
 * is c[]: computes the global element coordinates g[d] = c[d] + k[d] and
 * reports whether all of them are inside the tensor.  [D76] "The address
 * arithmetic moves into a descriptor" and the coordinate comment of "An exact
 * round trip": coordinates are element offsets, innermost dimension first.
 * [CDSL] "Describe the memory layout first": offset = row * cols + col for a
 * row-major matrix, strides counted per dimension.
 */
static int element_in_bounds(const oracle_view* v, const int32_t* c, uint64_t e,
                             int64_t* g)
{
    uint64_t rest = e;
    int inside = 1;
    for (int32_t d = 0; d < v->rank; ++d) {
        int64_t k = (int64_t)(rest % visits_along(v, d));
        rest /= visits_along(v, d);
        g[d] = (int64_t)c[d] + k * (int64_t)step_along(v, d);
        if (g[d] < 0 || g[d] >= (int64_t)v->dims[d]) inside = 0;
    }
    return inside;
}

static uint64_t element_address(const oracle_view* v, const int64_t* g)
{
    uint64_t addr = 0;
    for (int32_t d = 0; d < v->rank; ++d) addr += (uint64_t)g[d] * v->strides[d];
    return addr;
}

/*
 * Load: [L04] "What the issuing thread actually does" - the engine walks the
 * rectangular region the descriptor describes, reads it from global memory
 * and writes it into shared memory; [ARC] "The architecture": out-of-bounds
 * accesses are zero-filled (reading R1); the bytes land swizzled (R3).
 */
void oracle_tile_load(const oracle_view* v, const uint8_t* base,
                      const int32_t* coords, uint64_t n, uint8_t* packed)
{
    uint64_t box_bytes = oracle_box_bytes(v);
    uint64_t box_elems = box_bytes / (uint64_t)v->esize;
    int64_t g[ORACLE_MAX_RANK];
    for (uint64_t i = 0; i < n; ++i) {
        const int32_t* c = coords + i * (uint64_t)v->rank;
        uint8_t* image = packed + i * box_bytes;
        for (uint64_t e = 0; e < box_elems; ++e) {
            int inside = element_in_bounds(v, c, e, g);
            uint64_t addr = inside ? element_address(v, g) : 0;
            for (int32_t b = 0; b < v->esize; ++b) {
                uint64_t o = e * (uint64_t)v->esize + (uint64_t)b;
                image[oracle_swizzle(o, v->swizzle_bits)] = inside ? base[addr + (uint64_t)b] : 0;
            }
        }
    }
}

/*
 * Which image bytes a load fills rather than reads: [ARC] "The architecture:
 * every piece explained" (the engine fills what lies outside the tensor) and
 * reading R6.  Same walk as the load, recording "outside" at the swizzled
 * position of each byte of each element.
 */
void oracle_tile_oob_mask(const oracle_view* v, const int32_t* coords, uint64_t n,
                          uint8_t* mask)
{
    uint64_t box_bytes = oracle_box_bytes(v);
    uint64_t box_elems = box_bytes / (uint64_t)v->esize;
    int64_t g[ORACLE_MAX_RANK];
    for (uint64_t i = 0; i < n; ++i) {
        const int32_t* c = coords + i * (uint64_t)v->rank;
        uint8_t* image = mask + i * box_bytes;
        for (uint64_t e = 0; e < box_elems; ++e) {
            uint8_t outside = element_in_bounds(v, c, e, g) ? 0 : 1;
            for (int32_t b = 0; b < v->esize; ++b) {
                uint64_t o = e * (uint64_t)v->esize + (uint64_t)b;
                image[oracle_swizzle(o, v->swizzle_bits)] = outside;
            }
        }
    }
}

/*
 * Store: [L04] "Store completion - commit group and wait group" and [D76]
 * "Exercise"/"Solution": the shared-to-global direction writes the box image
 * back at the same coordinates; elements outside the tensor are not written
 * (reading R2).  Boxes are applied in list order.
 */
void oracle_tile_store(const oracle_view* v, uint8_t* base,
                       const int32_t* coords, uint64_t n, const uint8_t* packed)
{
    uint64_t box_bytes = oracle_box_bytes(v);
    uint64_t box_elems = box_bytes / (uint64_t)v->esize;
    int64_t g[ORACLE_MAX_RANK];
    for (uint64_t i = 0; i < n; ++i) {
        const int32_t* c = coords + i * (uint64_t)v->rank;
        const uint8_t* image = packed + i * box_bytes;
        for (uint64_t e = 0; e < box_elems; ++e) {
            if (!element_in_bounds(v, c, e, g)) continue;
            uint64_t addr = element_address(v, g);
            for (int32_t b = 0; b < v->esize; ++b) {
                uint64_t o = e * (uint64_t)v->esize + (uint64_t)b;
                base[addr + (uint64_t)b] = image[oracle_swizzle(o, v->swizzle_bits)];
            }
        }
    }
}

/* [D76] "Exercise": load every box, then write it back through a second map
 * with the same box shape. */
int32_t oracle_roundtrip(const oracle_view* src, const uint8_t* src_base,
                         const oracle_view* dst, uint8_t* dst_base,
                         const int32_t* coords, uint64_t n)
{
    if (src->rank != dst->rank || src->esize != dst->esize ||
        src->swizzle_bits != dst->swizzle_bits)
        return -1;
    for (int32_t d = 0; d < src->rank; ++d)
        if (src->box[d] != dst->box[d] || step_along(src, d) != step_along(dst, d)) return -1;
    uint64_t box_bytes = oracle_box_bytes(src);
    if (n == 0) return 0;
    uint8_t* packed = (uint8_t*)malloc(n * box_bytes);
    if (!packed) return -1;
    oracle_tile_load(src, src_base, coords, n, packed);
    oracle_tile_store(dst, dst_base, coords, n, packed);
    free(packed);
    return 0;
}

/*
 * [D76] "An exact round trip": the page's kernel adds 1.0f to every element
 * of the landed tile in shared memory; "Exercise"/"Solution" store the
 * updated tile back with the tensor store.  Elementwise, so the swizzled
 * order of the image does not matter.  Plain C float addition (binary32,
 * round to nearest even, no contraction).
 */
void oracle_add_f32(uint8_t* packed, uint64_t bytes, float addend)
{
    for (uint64_t o = 0; o + 4 <= bytes; o += 4) {
        float x;
        memcpy(&x, packed + o, 4);
        x = x + addend;
        memcpy(packed + o, &x, 4);
    }
}

int32_t oracle_roundtrip_add_f32(const oracle_view* src, const uint8_t* src_base,
                                 const oracle_view* dst, uint8_t* dst_base,
                                 const int32_t* coords, uint64_t n, float addend)
{
    if (src->esize != 4 || dst->esize != 4 || src->rank != dst->rank ||
        src->swizzle_bits != dst->swizzle_bits)
        return -1;
    for (int32_t d = 0; d < src->rank; ++d)
        if (src->box[d] != dst->box[d] || step_along(src, d) != step_along(dst, d)) return -1;
    uint64_t box_bytes = oracle_box_bytes(src);
    if (n == 0) return 0;
    uint8_t* packed = (uint8_t*)malloc(n * box_bytes);
    if (!packed) return -1;
    oracle_tile_load(src, src_base, coords, n, packed);
    oracle_add_f32(packed, n * box_bytes, addend);
    oracle_tile_store(dst, dst_base, coords, n, packed);
    free(packed);
    return 0;
}
