/*
 * A plain C host against include/pkv.h: the header compiles as C, the
 * library links without PyTorch, and the host-only entry points work with no
 * GPU (metadata builder, sizing, argument checks, status strings).
 * Prints "abi ok" and exits 0 on success.
 */
#include <stdio.h>
#include <string.h>

#include "pkv.h"

static int fail(const char* what) {
    printf("FAIL %s\n", what);
    return 1;
}

int main(void) {
    /* the flatten example ("Model execution", section "Code"): A a 5-token
       prefill chunk on block [7], B a decode at position 37 on [2, 9, 4], C 3
       new tokens after 32 cached on [11, 12, 3] */
    const int32_t computed[3] = {0, 37, 32}, scheduled[3] = {5, 1, 3};
    const int32_t offsets[4] = {0, 1, 4, 7};
    const int32_t ids[7] = {7, 2, 9, 4, 11, 12, 3};
    int32_t qsl[4], seq_lens[3], table[3 * 3], mq = 0, ms = 0;
    int64_t slots[9], pos[9];
    pkv_status st = pkv_build_metadata(3, computed, scheduled, offsets, ids, 16, 3, 9, qsl,
                                       seq_lens, table, slots, pos, &mq, &ms);
    if (st != PKV_OK) return fail("pkv_build_metadata");
    const int64_t want[9] = {112, 113, 114, 115, 116, 69, 48, 49, 50};
    if (memcmp(slots, want, sizeof(want)) != 0) return fail("slot_mapping");
    if (qsl[3] != 9 || seq_lens[1] != 38 || seq_lens[2] != 35 || mq != 5 || ms != 38)
        return fail("metadata");
    if (pkv_workspace_bytes(1, 32, 128, 1) != 0) return fail("pkv_workspace_bytes");
    if (strcmp(pkv_status_string(PKV_ERR_WORKSPACE), "PKV_ERR_WORKSPACE") != 0)
        return fail("pkv_status_string");
    /* host-checkable errors return before any CUDA call */
    if (pkv_write(NULL, NULL, NULL, 0, NULL, NULL, 4, 16, 8, 128, PKV_BF16, NULL, NULL) != PKV_OK)
        return fail("empty write");
    if (pkv_attention_varlen(NULL, NULL, NULL, NULL, NULL, NULL, NULL, NULL, 4, 1, 1, 1, 16, 8,
                             2, 96, 16, 0.1f, 1, 1, NULL, 0, NULL, 4, PKV_BF16, NULL) !=
        PKV_ERR_UNSUPPORTED)
        return fail("head_dim 96");
    if (pkv_cascade_splits(5, 0, 8, 2, 128, PKV_BF16, 0) != 0) return fail("cascade splits");
    printf("abi ok\n");
    return 0;
}
