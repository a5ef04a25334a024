/*
 * The C ABI from plain C: no Python, no torch.
 *
 *   abi_roundtrip host   encoder rule checks that need no GPU
 *   abi_roundtrip gpu    a 1000 x 700 fp16 round trip (64 x 32 boxes with
 *                        ragged edges), a listed gather, the listed store of
 *                        those images, the host-buffer round trip, the fp32
 *                        update, the allocation-free round trip, a ring-checked
 *                        launch and the device status, checked against the
 *                        expected bytes computed here (a full-grid round trip
 *                        reproduces its input; a gathered box holds the source
 *                        rows and zeros outside; a store writes only in-bounds
 *                        elements; the update adds 1.0f to every element)
 *
 * Exit status 0 on success; the first failed check is printed.
 */
#include <stdint.h>
#include <stdio.h>
#include <stdlib.h>
#include <string.h>

#include "atb.h"

/* Only the CUDA runtime calls this program needs (the library has its own). */
typedef int cudaError_t;
extern cudaError_t cudaMalloc(void** p, size_t n);
extern cudaError_t cudaFree(void* p);
extern cudaError_t cudaMemcpy(void* dst, const void* src, size_t n, int kind);
extern cudaError_t cudaMemset(void* p, int v, size_t n);
extern cudaError_t cudaDeviceSynchronize(void);
enum { H2D = 1, D2H = 2 };

static int failures = 0;
#define CHECK(cond, ...)                                  \
    do {                                                  \
        if (!(cond)) {                                    \
            fprintf(stderr, "FAIL %s:%d: ", __FILE__, __LINE__); \
            fprintf(stderr, __VA_ARGS__);                 \
            fprintf(stderr, "\n");                        \
            ++failures;                                   \
        }                                                 \
    } while (0)

static void host_checks(void)
{
    atb_tensor_map m;
    uint64_t dims[2] = {1024, 64}, strides[2] = {2, 2048};
    uint32_t box[2] = {64, 16};
    CHECK(atb_version() == ATB_VERSION, "version %d", atb_version());
    CHECK(atb_tensor_map_size() == sizeof(atb_tensor_map), "map size");
    CHECK(atb_encode_tiled(&m, ATB_F16, 6, (void*)0x10000, dims, strides, box, NULL, ATB_SWIZZLE_NONE,
                           ATB_L2_PROMO_NONE, ATB_OOB_ZERO) == ATB_ERR_RANK, "rank");
    CHECK(atb_encode_tiled(&m, ATB_F16, 2, (void*)0x10008, dims, strides, box, NULL, ATB_SWIZZLE_NONE,
                           ATB_L2_PROMO_NONE, ATB_OOB_ZERO) == ATB_ERR_BASE_ALIGN, "base alignment");
    strides[1] = 2040;
    CHECK(atb_encode_tiled(&m, ATB_F16, 2, (void*)0x10000, dims, strides, box, NULL, ATB_SWIZZLE_NONE,
                           ATB_L2_PROMO_NONE, ATB_OOB_ZERO) == ATB_ERR_STRIDE_ALIGN, "stride alignment");
    CHECK(strstr(atb_last_error(), "strides_bytes[1]") != NULL, "error text: %s", atb_last_error());
    strides[1] = 2048;
    box[1] = 300;
    CHECK(atb_encode_tiled(&m, ATB_F16, 2, (void*)0x10000, dims, strides, box, NULL, ATB_SWIZZLE_NONE,
                           ATB_L2_PROMO_NONE, ATB_OOB_ZERO) == ATB_ERR_BOX_DIM, "box extent");
    box[1] = 16;
    box[0] = 32;
    CHECK(atb_encode_tiled(&m, ATB_F16, 2, (void*)0x10000, dims, strides, box, NULL, ATB_SWIZZLE_128B,
                           ATB_L2_PROMO_NONE, ATB_OOB_ZERO) == ATB_ERR_SWIZZLE_SPAN, "swizzle span");
    CHECK(strcmp(atb_status_string(ATB_ERR_TIMEOUT), "ATB_ERR_TIMEOUT") == 0, "status string");
    CHECK(strcmp(atb_status_string(ATB_ERR_RING_CHECK), "ATB_ERR_RING_CHECK") == 0, "status string");
    CHECK(atb_box_bytes(NULL) == 0 && atb_grid_tiles(NULL) == 0, "NULL map queries");
    box[0] = 64;
    CHECK(atb_encode_tiled(&m, ATB_U8, 2, (void*)0x10000, dims, strides, box, NULL, ATB_SWIZZLE_NONE,
                           ATB_L2_PROMO_NONE, ATB_OOB_NAN) == ATB_ERR_DTYPE, "NaN fill of an integer type");
}

/* Next pseudo-random byte of a 64-bit linear congruential stream. */
static uint8_t next_byte(uint64_t* state)
{
    *state = *state * 6364136223846793005ull + 1442695040888963407ull;
    return (uint8_t)(*state >> 56);
}

static int gpu_checks(void)
{
    const uint64_t cols = 1000, rows = 700, pitch = 2016; /* fp16, 16 padding bytes per row */
    const size_t nbytes = pitch * rows;
    uint8_t* h_src = malloc(nbytes);
    uint8_t* h_out = malloc(nbytes);
    uint64_t state = 0x9E3779B97F4A7C15ull;
    for (size_t i = 0; i < nbytes; ++i) h_src[i] = next_byte(&state);
    void *d_src = NULL, *d_dst = NULL, *d_packed = NULL, *d_coords = NULL;
    CHECK(cudaMalloc(&d_src, nbytes) == 0 && cudaMalloc(&d_dst, nbytes) == 0, "cudaMalloc");
    cudaMemcpy(d_src, h_src, nbytes, H2D);
    cudaMemcpy(d_dst, h_src, nbytes, H2D); /* padding bytes equal: the whole buffer must match */
    for (uint64_t r = 0; r < 10; ++r)      /* ... once the round trip rewrites these elements */
        cudaMemset((uint8_t*)d_dst + r * pitch, 0, cols * 2);

    atb_tensor_map ms, md;
    uint64_t dims[2] = {cols, rows}, strides[2] = {2, pitch};
    uint32_t box[2] = {64, 32};
    atb_status st = atb_encode_tiled(&ms, ATB_F16, 2, d_src, dims, strides, box, NULL, ATB_SWIZZLE_NONE,
                                     ATB_L2_PROMO_NONE, ATB_OOB_ZERO);
    CHECK(st == ATB_OK, "encode source: %s %s", atb_status_string(st), atb_last_error());
    st = atb_encode_tiled(&md, ATB_F16, 2, d_dst, dims, strides, box, NULL, ATB_SWIZZLE_NONE, ATB_L2_PROMO_NONE,
                          ATB_OOB_ZERO);
    CHECK(st == ATB_OK, "encode destination: %s", atb_status_string(st));
    CHECK(atb_grid_tiles(&ms) == 16 * 22, "grid boxes %llu", (unsigned long long)atb_grid_tiles(&ms));
    st = atb_tile_roundtrip(&ms, &md, NULL, 0, NULL, NULL);
    CHECK(st == ATB_OK, "round trip: %s %s", atb_status_string(st), atb_last_error());
    atb_device_report rep;
    CHECK(atb_device_status(NULL, &rep) == ATB_OK && rep.errors == 0, "device status %d", rep.code);
    cudaMemcpy(h_out, d_dst, nbytes, D2H);
    CHECK(memcmp(h_out, h_src, nbytes) == 0, "round trip differs from its input");

    /* gather two listed boxes, one hanging over the top-left corner */
    int32_t coords[4] = {128, 64, -32, -8};
    const size_t bb = atb_box_bytes(&ms);
    CHECK(bb == 64 * 32 * 2, "box bytes %zu", bb);
    cudaMalloc(&d_packed, 2 * bb);
    cudaMalloc(&d_coords, sizeof coords);
    cudaMemcpy(d_coords, coords, sizeof coords, H2D);
    st = atb_tile_load(&ms, (const int32_t*)d_coords, 2, d_packed, NULL, NULL);
    CHECK(st == ATB_OK, "gather: %s", atb_status_string(st));
    uint8_t* img = malloc(2 * bb);
    cudaMemcpy(img, d_packed, 2 * bb, D2H);
    for (int b = 0; b < 2; ++b)
        for (int r = 0; r < 32; ++r)
            for (int x = 0; x < 64; ++x) {
                const int64_t gy = coords[2 * b + 1] + r, gx = coords[2 * b] + x;
                uint16_t want = 0, got;
                if (gx >= 0 && gy >= 0 && gx < (int64_t)cols && gy < (int64_t)rows)
                    memcpy(&want, h_src + gy * pitch + gx * 2, 2);
                memcpy(&got, img + b * bb + (size_t)(r * 64 + x) * 2, 2);
                if (got != want) {
                    CHECK(0, "box %d row %d col %d: got %u want %u", b, r, x, got, want);
                    b = 2; r = 32; break;
                }
            }
    CHECK(atb_device_status(NULL, &rep) == ATB_OK, "device status after gather %d", rep.code);

    /* store the two images into a tensor filled with 0xAB: in-bounds elements
       take the image, everything else keeps the fill (the corner box starts
       before the tensor, so it is written with clipped thread stores) */
    cudaMemset(d_dst, 0xAB, nbytes);
    st = atb_tile_store(&md, (const int32_t*)d_coords, 2, d_packed, NULL, NULL);
    CHECK(st == ATB_OK, "store: %s", atb_status_string(st));
    CHECK(atb_device_status(NULL, &rep) == ATB_OK, "device status after store %d", rep.code);
    cudaMemcpy(h_out, d_dst, nbytes, D2H);
    for (uint64_t y = 0; y < rows; ++y)
        for (uint64_t x = 0; x < pitch / 2; ++x) {
            uint16_t want = 0xABAB, got;
            for (int b = 0; b < 2; ++b) {
                const int64_t ry = (int64_t)y - coords[2 * b + 1], rx = (int64_t)x - coords[2 * b];
                if (x < cols && ry >= 0 && ry < 32 && rx >= 0 && rx < 64) memcpy(&want, h_src + y * pitch + x * 2, 2);
            }
            memcpy(&got, h_out + y * pitch + x * 2, 2);
            if (got != want) {
                CHECK(0, "store: row %llu col %llu: got %u want %u", (unsigned long long)y, (unsigned long long)x,
                      got, want);
                y = rows;
                break;
            }
        }

    /* host-resident round trip: pageable host buffers in, host buffer out */
    uint8_t* h_back = malloc(nbytes);
    memset(h_back, 0, nbytes);
    st = atb_tile_roundtrip_host(&ms, &md, h_src, h_back, 5, NULL, NULL);
    CHECK(st == ATB_OK, "host round trip: %s %s", atb_status_string(st), atb_last_error());
    cudaDeviceSynchronize();
    CHECK(atb_device_status(NULL, &rep) == ATB_OK, "device status after host round trip %d", rep.code);
    for (uint64_t y = 0; y < rows; ++y)
        if (memcmp(h_back + y * pitch, h_src + y * pitch, cols * 2) != 0) {
            CHECK(0, "host round trip: row %llu differs", (unsigned long long)y);
            break;
        }

    /* fp32 update over the same storage seen as 500 x 700 fp32 with finite values */
    float* h_f = malloc(nbytes);
    for (size_t i = 0; i < nbytes / 4; ++i) {
        uint32_t bits = 0;
        for (int k = 0; k < 4; ++k) bits = (bits << 8) | next_byte(&state);
        if ((bits & 0x7F800000u) == 0x7F800000u) bits &= 0xBFFFFFFFu; /* no Inf or NaN */
        memcpy(&h_f[i], &bits, 4);
    }
    cudaMemcpy(d_src, h_f, nbytes, H2D);
    atb_tensor_map fs, fd;
    uint64_t fdims[2] = {cols / 2, rows};
    uint32_t fbox[2] = {32, 64};
    st = atb_encode_tiled(&fs, ATB_F32, 2, d_src, fdims, strides, fbox, NULL, ATB_SWIZZLE_128B, ATB_L2_PROMO_NONE,
                          ATB_OOB_ZERO);
    CHECK(st == ATB_OK, "encode fp32 source: %s", atb_last_error());
    st = atb_encode_tiled(&fd, ATB_F32, 2, d_dst, fdims, strides, fbox, NULL, ATB_SWIZZLE_128B, ATB_L2_PROMO_NONE,
                          ATB_OOB_ZERO);
    CHECK(st == ATB_OK, "encode fp32 destination: %s", atb_last_error());
    st = atb_tile_roundtrip_add_f32(&fs, &fd, NULL, 0, 1.0f, NULL, NULL);
    CHECK(st == ATB_OK, "fp32 update: %s", atb_status_string(st));
    CHECK(atb_device_status(NULL, &rep) == ATB_OK, "device status after fp32 update %d", rep.code);
    float* h_g = malloc(nbytes);
    cudaMemcpy(h_g, d_dst, nbytes, D2H);
    for (uint64_t y = 0; y < rows; ++y)
        for (uint64_t x = 0; x < cols / 2; ++x) {
            const float want = h_f[y * (pitch / 4) + x] + 1.0f;
            const float got = h_g[y * (pitch / 4) + x];
            if (memcmp(&want, &got, 4) != 0) {
                CHECK(0, "fp32 update: row %llu col %llu", (unsigned long long)y, (unsigned long long)x);
                y = rows;
                break;
            }
        }

    /* allocation-free round trip with the ring check on, back over the fp16 maps */
    cudaMemcpy(d_src, h_src, nbytes, H2D);
    cudaMemset(d_dst, 0, nbytes);
    atb_launch checked;
    memset(&checked, 0, sizeof checked);
    checked.checks = ATB_CHECK_RING;
    st = atb_tile_roundtrip_noalloc(&ms, &md, NULL, 0, &checked, NULL, &rep);
    CHECK(st == ATB_OK && rep.errors == 0, "allocation-free round trip: %s, %u errors", atb_status_string(st),
          rep.errors);
    cudaMemcpy(h_out, d_dst, nbytes, D2H);
    for (uint64_t y = 0; y < rows; ++y)
        if (memcmp(h_out + y * pitch, h_src + y * pitch, cols * 2) != 0) {
            CHECK(0, "allocation-free round trip: row %llu differs", (unsigned long long)y);
            break;
        }

    cudaFree(d_src); cudaFree(d_dst); cudaFree(d_packed); cudaFree(d_coords);
    free(h_src); free(h_out); free(img); free(h_back); free(h_f); free(h_g);
    return failures;
}

int main(int argc, char** argv)
{
    host_checks();
    if (argc > 1 && strcmp(argv[1], "gpu") == 0) gpu_checks();
    if (failures) {
        fprintf(stderr, "%d check(s) failed\n", failures);
        return 1;
    }
    printf("ok\n");
    return 0;
}
