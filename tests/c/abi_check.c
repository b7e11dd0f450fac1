/*
 * A plain C host program against include/mqa.h, linked with libmqa.so: it
 * checks that the header compiles as C, that every call links, and that the
 * host-side validation answers without a GPU.  Test infrastructure: built and
 * run by tests/test_c_program.py.
 */
#include <stdio.h>
#include <string.h>

#include "mqa.h"

static int failures = 0;

static void expect(const char *what, mqa_status got, mqa_status want)
{
    if (got != want) {
        printf("FAIL %s: got %s, want %s (%s)\n", what, mqa_status_string(got),
               mqa_status_string(want), mqa_last_error_message());
        ++failures;
    }
}

int main(void)
{
    /* a 16-byte aligned stand-in address; the calls below reject their
     * arguments on the host and never dereference it */
    static char buf[64] __attribute__((aligned(16)));
    void *p = buf;
    float *f = (float *)buf;
    int32_t *i = (int32_t *)buf;

    if (strcmp(mqa_status_string(MQA_ERR_TIMEOUT), "MQA_ERR_TIMEOUT") != 0) {
        printf("FAIL status string\n");
        ++failures;
    }
    expect("dense D=96", mqa_logits(p, p, f, f, i, i, f, 4, 256, 64, 96, 256, MQA_CLEAN, NULL),
           MQA_ERR_UNSUPPORTED);
    expect("dense ldo < S_kv", mqa_logits(p, p, f, f, i, i, f, 4, 256, 64, 128, 255, MQA_CLEAN, NULL),
           MQA_ERR_INVALID_ARG);
    expect("dense S_q = 0", mqa_logits(NULL, NULL, NULL, NULL, NULL, NULL, NULL, 0, 256, 64, 128, 256,
                                       MQA_CLEAN, NULL),
           MQA_OK);
    expect("metadata block_kv", paged_mqa_logits_metadata(i, 2, 2, 48, 8, i, NULL),
           MQA_ERR_UNSUPPORTED);
    expect("paged H=8", paged_mqa_logits(p, p, f, f, i, i, 16, i, f, 2, 2, 8, 128, 64, 40, 8, 1024,
                                         MQA_CLEAN, NULL),
           MQA_ERR_UNSUPPORTED);
    expect("paged compressed", paged_mqa_logits(p, p, f, f, i, i, 16, i, f, 2, 2, 64, 128, 64, 40, 8,
                                                1024, MQA_CLEAN | MQA_COMPRESSED, NULL),
           MQA_ERR_UNSUPPORTED);
    expect("paged fused with scales", paged_mqa_logits(p, p, f, f, i, i, 16, i, f, 2, 2, 64, 128, 64,
                                                       40, 8, 1024, MQA_CLEAN | MQA_KV_FUSED, NULL),
           MQA_ERR_INVALID_ARG);
    expect("noalloc ldo", paged_mqa_logits_noalloc(p, p, f, f, i, i, 16, f, 2, 2, 64, 128, 64, 40,
                                                   1000, MQA_CLEAN, NULL),
           MQA_ERR_INVALID_ARG);
    expect("topk k=0", mqa_topk_indices(f, i, i, i, 4, 256, 256, 0, 0, NULL), MQA_ERR_INVALID_ARG);
    expect("paged topk width", paged_mqa_topk_indices(f, i, i, 2, 2, 1024, 1000, 16, NULL),
           MQA_ERR_INVALID_ARG);
    {
        /* fused logits + top-k: the workspace size is a pure function; the
         * call rejects a short workspace, a clean flag and topk = 0 */
        const size_t ws = mqa_logits_topk_workspace_size(4, 256);
        if (ws == 0 || ws != mqa_logits_topk_workspace_size(4, 256) ||
            mqa_logits_topk_workspace_size(-1, 256) != 0) {
            printf("FAIL fused workspace size %zu\n", ws);
            ++failures;
        }
        static char wsbuf[256] __attribute__((aligned(256)));
        expect("fused short workspace",
               mqa_logits_topk(p, p, f, f, i, i, i, wsbuf, 256, 4, 256, 64, 128, 16, 0, NULL),
               MQA_ERR_INVALID_ARG);
        expect("fused clean flag",
               mqa_logits_topk(p, p, f, f, i, i, i, wsbuf, ws, 4, 256, 64, 128, 16, MQA_CLEAN, NULL),
               MQA_ERR_INVALID_ARG);
        expect("fused topk=0",
               mqa_logits_topk(p, p, f, f, i, i, i, wsbuf, ws, 4, 256, 64, 128, 0, 0, NULL),
               MQA_ERR_INVALID_ARG);
        expect("fused S_q = 0",
               mqa_logits_topk(NULL, NULL, NULL, NULL, NULL, NULL, NULL, NULL, 0, 0, 256, 64, 128,
                               16, 0, NULL),
               MQA_OK);
    }
    {
        const uint32_t *u = (const uint32_t *)buf;
        expect("mx D=64", mqa_logits_mx(p, u, p, u, f, i, i, f, 4, 256, 64, 64, 256, MQA_CLEAN, NULL),
               MQA_ERR_UNSUPPORTED);
        expect("mxfp4 alignment", mqa_logits_mx(p, u, p, u, f, i, i, f, 4, 256, 64, 128, 256,
                                                MQA_CLEAN | MQA_MXFP4, NULL),
               MQA_ERR_INVALID_ARG);
        expect("paged mx D=64", paged_mqa_logits_mx(p, u, p, u, f, i, i, 16, i, f, 2, 2, 64, 64, 64,
                                                    40, 8, 1024, MQA_CLEAN, NULL),
               MQA_ERR_UNSUPPORTED);
        expect("paged mx null q_sf", paged_mqa_logits_mx(p, NULL, p, u, f, i, i, 16, i, f, 2, 2, 64,
                                                         128, 64, 40, 8, 1024, MQA_CLEAN, NULL),
               MQA_ERR_INVALID_ARG);
        expect("scheduled null meta", mqa_logits_scheduled(p, p, f, f, i, i, NULL, 8, f, 4, 256, 64,
                                                           128, 256, MQA_CLEAN, NULL),
               MQA_ERR_INVALID_ARG);
        expect("dense metadata H=16", mqa_logits_metadata(i, i, 4, 256, 16, 8, i, NULL),
               MQA_ERR_UNSUPPORTED);
        expect("dense unknown flag", mqa_logits(p, p, f, f, i, i, f, 4, 256, 64, 128, 256, 128u, NULL),
               MQA_ERR_INVALID_ARG);
        expect("bf16 weights misaligned", mqa_logits(p, p, f, (const char *)buf + 8, i, i, f, 4, 256,
                                                     64, 128, 256, MQA_CLEAN | MQA_WEIGHTS_BF16, NULL),
               MQA_ERR_INVALID_ARG);
    }
    expect("wait limit", mqa_set_wait_limit(0), MQA_OK);
    if (failures == 0)
        printf("abi_check: ok\n");
    return failures == 0 ? 0 : 1;
}
