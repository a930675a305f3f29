/* A plain C99 client of the qgemv C ABI: no Python, no torch, no CUDA headers.
 *
 *   abi_client <fmt> <n_out> <n_in> <W.f32> <canonical.out> <packed.out>
 *
 * reads an fp32 [n_out][n_in] matrix, quantizes it (qg_quantize), converts the
 * canonical bytes to the device layout (qg_to_device_layout), packs the matrix
 * in one step (qg_pack) and writes the canonical and device-layout bytes.  It
 * checks on the way that the sizes agree, that qg_pack gives the two-step
 * bytes, and that calls with bad arguments are refused before any launch.
 * Exit status 0 on success; a message on stderr and status 1 otherwise. */
#include "qgemv.h"

#include <stdio.h>
#include <stdlib.h>
#include <string.h>

static int fail(const char* what) {
    fprintf(stderr, "abi_client: %s\n", what);
    return 1;
}

static qg_fmt parse_fmt(const char* s, int* ok) {
    *ok = 1;
    if (strcmp(s, "q8_0") == 0) return QG_Q8_0;
    if (strcmp(s, "q4_0") == 0) return QG_Q4_0;
    if (strcmp(s, "affine4_g64") == 0) return QG_AFFINE4_G64;
    if (strcmp(s, "bf16") == 0) return QG_BF16;
    if (strcmp(s, "q5_0") == 0) return QG_Q5_0;
    *ok = 0;
    return QG_Q8_0;
}

static int write_file(const char* path, const void* p, size_t n) {
    FILE* f = fopen(path, "wb");
    size_t w;
    if (!f) return 0;
    w = fwrite(p, 1, n, f);
    return fclose(f) == 0 && w == n;
}

int main(int argc, char** argv) {
    qg_fmt fmt;
    int ok;
    int64_t n_out, n_in;
    size_t n_w, canon_bytes, packed_bytes;
    float* W;
    unsigned char *canon, *packed, *packed1;
    FILE* f;
    int rc = 0;

    if (argc != 7) return fail("usage: abi_client fmt n_out n_in W.f32 canonical.out packed.out");
    if (qg_abi_version() != 1) return fail("unexpected ABI version");
    fmt = parse_fmt(argv[1], &ok);
    if (!ok) return fail("unknown format");
    n_out = strtoll(argv[2], NULL, 10);
    n_in = strtoll(argv[3], NULL, 10);
    canon_bytes = qg_canonical_bytes(fmt, n_out, n_in);
    packed_bytes = qg_packed_bytes(fmt, n_out, n_in);
    if (canon_bytes == 0 || packed_bytes < canon_bytes) return fail("sizes");
    if ((size_t)qg_row_stride(fmt, n_in) * (size_t)n_out != packed_bytes) return fail("row stride");

    n_w = (size_t)n_out * (size_t)n_in;
    W = (float*)malloc(n_w * sizeof(float));
    canon = (unsigned char*)malloc(canon_bytes);
    packed = (unsigned char*)malloc(packed_bytes);
    packed1 = (unsigned char*)malloc(packed_bytes);
    if (!W || !canon || !packed || !packed1) return fail("out of host memory");
    f = fopen(argv[4], "rb");
    if (!f || fread(W, sizeof(float), n_w, f) != n_w) return fail("cannot read W");
    fclose(f);

    if (qg_quantize(fmt, W, n_out, n_in, canon) != QG_OK) rc = fail("qg_quantize");
    if (!rc && qg_to_device_layout(fmt, canon, n_out, n_in, packed) != QG_OK) rc = fail("qg_to_device_layout");
    if (!rc && qg_pack(fmt, W, n_out, n_in, packed1) != QG_OK) rc = fail("qg_pack");
    if (!rc && memcmp(packed, packed1, packed_bytes) != 0) rc = fail("qg_pack differs from the two steps");

    /* refused before any launch: null pointers, ntok out of range, a ragged n_in */
    if (!rc && qg_quantize(fmt, NULL, n_out, n_in, canon) != QG_EINVAL) rc = fail("null W accepted");
    if (!rc && qg_pack(fmt, W, n_out, n_in + 1, packed1) != QG_EINVAL) rc = fail("ragged n_in accepted");
    if (!rc && qgemv(fmt, NULL, n_out, n_in, NULL, NULL, 1, NULL) != QG_EINVAL) rc = fail("null qgemv accepted");
    if (!rc && qgemv(fmt, packed, n_out, n_in, W, W, 5, NULL) != QG_EINVAL) rc = fail("ntok 5 accepted");
    if (!rc && strcmp(qg_strerror(QG_OK), qg_strerror(QG_EINVAL)) == 0) rc = fail("status strings");

    if (!rc && !write_file(argv[5], canon, canon_bytes)) rc = fail("cannot write canonical bytes");
    if (!rc && !write_file(argv[6], packed, packed_bytes)) rc = fail("cannot write packed bytes");
    free(W);
    free(canon);
    free(packed);
    free(packed1);
    return rc;
}
