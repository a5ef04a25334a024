/*
 * Plain CPU oracle for tiled tensor movement (test infrastructure only).
 *
 * This header and oracle.c are the checker, not the product: only the test
 * suite, the smoke check and the benchmark's CPU-baseline leg load them.  They
 * share no code, header, table or constant with the CUDA library; they state
 * the method from its definition so that a reader can compare them with the
 * pages by eye.
 *
 * Conventions (all from the pages, see oracle.c for the citations):
 *   - dims[], box[] and coordinates are innermost (contiguous) dimension first.
 *   - strides[d] is the byte distance between neighbours along dimension d;
 *     strides[0] must equal the element size (the innermost dimension is
 *     implicitly contiguous).
 *   - the packed image of tile i occupies bytes [i*box_bytes, (i+1)*box_bytes)
 *     and holds the box exactly as it sits in a shared-memory stage whose base
 *     is aligned to the swizzle pattern's period.
 */
#ifndef ORACLE_H
#define ORACLE_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define ORACLE_MAX_RANK 5

typedef struct {
    int32_t  rank;                      /* 1..5 */
    int32_t  esize;                     /* element size in bytes */
    int32_t  swizzle_bits;              /* B of Swizzle<B,4,3>: 0 none, 1 32B, 2 64B, 3 128B */
    int32_t  pad_;
    uint64_t dims[ORACLE_MAX_RANK];     /* extent per dimension, innermost first */
    uint64_t strides[ORACLE_MAX_RANK];  /* byte stride per dimension, innermost first */
    uint32_t box[ORACLE_MAX_RANK];      /* box extent per dimension, innermost first */
    uint32_t estr[ORACLE_MAX_RANK];     /* traversal step per dimension (0 or 1 = every element) */
} oracle_view;

/* Swizzle<B,4,3> applied to a byte offset inside a box image. */
uint64_t oracle_swizzle(uint64_t offset, int32_t bits);

/* Bytes of one box image: the element size times, per dimension, the number
 * of elements the box visits (ceil(box / step)). */
uint64_t oracle_box_bytes(const oracle_view* v);

/* Number of boxes that tile the whole tensor (edge boxes included). */
uint64_t oracle_grid_count(const oracle_view* v);

/* Origins of the grid boxes, tile index t -> coords[t*rank .. t*rank+rank-1]. */
void oracle_grid_coords(const oracle_view* v, int32_t* coords);

/* Gather n boxes at the given origins into the packed image buffer. */
void oracle_tile_load(const oracle_view* v, const uint8_t* base,
                      const int32_t* coords, uint64_t n, uint8_t* packed);

/* Marks, for n boxes, which bytes of each packed image belong to elements
 * outside the tensor: mask[i*box_bytes + swizzled offset] = 1 for every byte
 * of an out-of-bounds element, 0 otherwise.  These are the bytes a load fills
 * instead of reading. */
void oracle_tile_oob_mask(const oracle_view* v, const int32_t* coords, uint64_t n,
                          uint8_t* mask);

/* Scatter n packed box images back to the tensor; out-of-bounds elements are skipped. */
void oracle_tile_store(const oracle_view* v, uint8_t* base,
                       const int32_t* coords, uint64_t n, const uint8_t* packed);

/* store(dst, coords, load(src, coords)); returns 0, or -1 if the box shapes,
 * element sizes or swizzle modes of the two views differ or memory runs out. */
int32_t oracle_roundtrip(const oracle_view* src, const uint8_t* src_base,
                         const oracle_view* dst, uint8_t* dst_base,
                         const int32_t* coords, uint64_t n);

/* Adds `addend` to every fp32 element of `bytes` bytes of packed images, in
 * place (IEEE binary32, round to nearest even). */
void oracle_add_f32(uint8_t* packed, uint64_t bytes, float addend);

/* store(dst, coords, load(src, coords) + addend) for fp32 views; returns 0,
 * or -1 on mismatched views, a non-4-byte element or out of memory. */
int32_t oracle_roundtrip_add_f32(const oracle_view* src, const uint8_t* src_base,
                                 const oracle_view* dst, uint8_t* dst_base,
                                 const int32_t* coords, uint64_t n, float addend);

#ifdef __cplusplus
}
#endif

#endif
