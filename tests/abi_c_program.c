/* A plain C99 program against include/pagedkv.h: the header must compile as
 * C, and every entry point must link from libpagedkv.so with C linkage.  It
 * runs only the calls that need no GPU (status strings, sizes, host-side
 * argument checks).  Built and run by tests/test_abi.py. */
#include <stdio.h>
#include <string.h>

#include "pagedkv.h"

int main(void) {
    /* every entry point, taken by address so that the linker must resolve it */
    const void* entry[] = {
        (const void*)pkv_status_string, (const void*)pkv_version, (const void*)paged_kv_append,
        (const void*)paged_attention_workspace_bytes, (const void*)paged_attention_plan,
        (const void*)paged_attention_partition_size, (const void*)paged_attention_decode,
        (const void*)paged_attention_append_decode, (const void*)paged_attention_decode_grouped,
        (const void*)paged_attention_append_decode_grouped,
        (const void*)paged_attention_grouped_workspace_bytes, (const void*)paged_attention_decode_static,
        (const void*)copy_blocks, (const void*)swap_blocks, (const void*)compact_tokens,
        (const void*)pkv_check_device_error, (const void*)pkv_launch_count, (const void*)pkv_wait_selftest};
    size_t i;
    pkv_cache_desc desc;
    for (i = 0; i < sizeof(entry) / sizeof(entry[0]); ++i)
        if (!entry[i]) return 2;
    if (strcmp(pkv_status_string(PKV_OK), "ok") != 0) return 3;
    if (paged_attention_workspace_bytes(8, 64, 128, 512, 0) != 0) return 4; /* one partition: no workspace */
    if (paged_attention_workspace_bytes(8, 64, 128, 131072, 0) == 0) return 5;
    desc.num_blocks = 64;
    desc.num_kv_heads = 1;
    desc.block_size = 24; /* not 16 or 32: rejected before any CUDA call */
    desc.head_dim = 128;
    desc.dtype = PKV_BF16;
    if (paged_attention_decode((void*)16, (void*)16, (void*)16, (const int32_t*)16, 4, (const int32_t*)16, 1, 4, 16,
                               0.1f, (void*)16, PKV_FP32, &desc, 0, NULL, 0, NULL) != PKV_ERR_UNSUPPORTED)
        return 6;
    if (paged_kv_append(NULL, NULL, NULL, 0, NULL, NULL, NULL, NULL) != PKV_ERR_INVALID_ARG) return 7;
    if (pkv_wait_selftest(0, NULL) != PKV_ERR_INVALID_ARG) return 8; /* limit out of range: nothing launched */
    if (pkv_wait_selftest(2000001, NULL) != PKV_ERR_INVALID_ARG) return 9;
    printf("c abi ok, version %d\n", pkv_version());
    return 0;
}
