/* A plain C caller of the library: includes only include/sdv2.h, links libsdv2.so, and checks
 * the host-side contract that needs no GPU (size queries, the visible-token formula, argument
 * validation with status and message, status strings).  Exit code 0 = all checks passed. */
#include <stdint.h>
#include <stdio.h>
#include <string.h>

#include "sdv2.h"

static int failures = 0;
#define CHECK(cond)                                                         \
    do {                                                                    \
        if (!(cond)) {                                                      \
            fprintf(stderr, "check failed at line %d: %s\n", __LINE__, #cond); \
            ++failures;                                                     \
        }                                                                   \
    } while (0)

int main(void)
{
    /* the Wan-1.3B 480p stream: 12 heads, 30x52 tokens per frame, chunks of 3 frames,
       sink of 3 frames and a window of 18 */
    sdv2_stream_cfg c;
    memset(&c, 0, sizeof(c));
    c.batch = 1; c.heads = 12; c.head_dim = 128; c.rope_t = 44; c.rope_h = 42; c.rope_w = 42;
    c.rope_base = 10000.0; c.grid_h = 30; c.grid_w = 52; c.chunk_frames = 3; c.sink_frames = 3;
    c.window_frames = 18; c.refresh_chunks = 0; c.qkv_token_stride = 0;

    const size_t rows = (size_t)(3 + 18) * 1560;
    CHECK(sdv2_cache_bytes(&c) == (size_t)12 * rows * 128 * 2);
    CHECK(sdv2_meta_bytes(&c) == (size_t)21 * sizeof(sdv2_slot_meta));
    CHECK(sizeof(sdv2_slot_meta) == 16);
    CHECK(sdv2_workspace_bytes(&c) > 0);
    /* n = (c+1)*F frames appended; n_vis = min(F_s, n) + min(W, max(0, n - F_s)) */
    CHECK(sdv2_visible_tokens(&c, 0) == 3 * 1560);
    CHECK(sdv2_visible_tokens(&c, 1) == 6 * 1560);
    CHECK(sdv2_visible_tokens(&c, 6) == 21 * 1560);
    CHECK(sdv2_visible_tokens(&c, 1000) == 21 * 1560);
    CHECK(sdv2_visible_tokens(&c, -1) == -1);

    /* invalid configurations: every size query gives 0 */
    sdv2_stream_cfg bad = c;
    bad.rope_t = 43; bad.rope_h = 43;                    /* odd segments */
    CHECK(sdv2_cache_bytes(&bad) == 0 && sdv2_workspace_bytes(&bad) == 0);
    bad = c; bad.window_frames = 2;                      /* W < F */
    CHECK(sdv2_meta_bytes(&bad) == 0);

    /* argument validation: rejected before anything touches a device */
    void* fake = (void*)(uintptr_t)(1u << 20);
    int64_t start = 0, chunk = 0;
    CHECK(sdv2_rope_append_kv(&c, &start, &chunk, NULL, fake, fake, fake, fake, fake, fake, fake, NULL) ==
          SDV2_ERR_INVALID_ARG);
    CHECK(strlen(sdv2_last_error()) > 0);
    int64_t neg = -1;
    CHECK(sdv2_chunk_attention(&c, &neg, fake, fake, fake, 0.0f, fake, NULL, fake, NULL) == SDV2_ERR_INVALID_ARG);
    bad = c; bad.head_dim = 64; bad.rope_t = 22; bad.rope_h = 22; bad.rope_w = 20;
    CHECK(sdv2_chunk_attention(&bad, &chunk, fake, fake, fake, 0.0f, fake, NULL, fake, NULL) ==
          SDV2_ERR_UNSUPPORTED);
    CHECK(sdv2_motion_l2((const uint8_t*)fake, 1, 0, 4, 4, 1, (uint64_t*)fake, NULL, NULL) == SDV2_ERR_INVALID_ARG);

    CHECK(strcmp(sdv2_status_string(SDV2_OK), "ok") == 0);
    CHECK(sdv2_status_string(SDV2_ERR_TIMEOUT) != NULL);

    if (failures) return 1;
    printf("C ABI: all host-side checks passed\n");
    return 0;
}
