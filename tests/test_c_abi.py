"""The boundary as a C program sees it: the header compiles as strict C11
(gcc -std=c11 -Wall -Wextra -Werror -pedantic), the program links against
the library, and the host-only entry points behave as declared (layout,
shard bounds, accounting, buckets, the SM cap, the host Adam, status
strings).  No CUDA call is made, so this runs without a GPU."""
import os
import shutil
import subprocess

import pytest

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(HERE)

C_PROGRAM = r"""
#include <math.h>
#include <stdio.h>
#include <string.h>

#include "zero_step.h"

#define CHECK(cond)                                                   \
    do {                                                              \
        if (!(cond)) {                                                \
            fprintf(stderr, "line %d: %s\n", __LINE__, #cond);        \
            return 1;                                                 \
        }                                                             \
    } while (0)

int main(void)
{
    /* three tensors of 3, 5 and 7 elements over 4 ranks: M = 4 */
    const int64_t numel[3] = {3, 5, 7};
    zero_layout_t L;
    memset(&L, 0, sizeof L);
    CHECK(zero_init_layout(numel, 3, 4, 2, &L) == ZERO_OK);
    CHECK(L.N == 15 && L.M == 4 && L.P == 4);
    CHECK(L.shard_begin[3] == 12 && L.shard_end[3] == 15);
    int64_t covered = 0;
    for (int64_t s = 0; s < L.n_segs; ++s) covered += L.segs[s].len;
    CHECK(covered == 15 && L.seg_offsets[4] == L.n_segs);
    zero_free_layout(&L);
    zero_free_layout(&L); /* a freed table is accepted */
    CHECK(zero_init_layout(numel, 3, 0, 2, &L) == ZERO_EINVAL);

    int64_t b = -1, e = -1;
    CHECK(zero_shard_range(5, 4, 3, &b, &e) == ZERO_OK && b == 5 && e == 5); /* empty trailing shard */
    CHECK(zero_shard_range(5, 4, 4, &b, &e) == ZERO_EINVAL);

    /* 7.5 billion parameters on 64 ranks: 120 GB for plain data parallel */
    double bytes = 0.0;
    CHECK(zero_memory_bytes(7500000000LL, 64, 0, &bytes, NULL, NULL) == ZERO_OK);
    CHECK(fabs(bytes - 1.2e11) < 1.0);
    CHECK(zero_memory_bytes(7500000000LL, 64, 3, &bytes, NULL, NULL) == ZERO_OK);
    CHECK(fabs(bytes - 16.0 * 7500000000.0 / 64.0) < 1.0);

    /* buckets, two-call pattern, backward order */
    int32_t nb = 0;
    CHECK(zero_plan_buckets(numel, 3, 6, 1, NULL, 0, &nb) == ZERO_OK && nb == 2);
    zero_bucket_t bk[2];
    CHECK(zero_plan_buckets(numel, 3, 6, 1, bk, 2, &nb) == ZERO_OK);
    CHECK(bk[0].begin == 8 && bk[0].end == 15 && bk[1].begin == 0 && bk[1].end == 8);

    int32_t prev = -1;
    CHECK(zero_set_step_max_sms(7, &prev) == ZERO_OK);
    CHECK(zero_set_step_max_sms(-1, &prev) == ZERO_EINVAL);
    CHECK(zero_set_step_max_sms(0, &prev) == ZERO_OK && prev == 7);

    /* host Adam, first step from zero moments: each weight moves by about
       lr against the sign of its gradient (lr g / (|g| + eps)) */
    enum { n = 1000 };
    static uint16_t g16[n], p16[n];
    static float w[n], m[n], v[n];
    for (int i = 0; i < n; ++i) {
        g16[i] = (uint16_t)((i % 2 ? 0x8000u : 0u) | 0x1400u); /* +-2^-10 */
        w[i] = 0.5f;
        m[i] = 0.0f;
        v[i] = 0.0f;
    }
    CHECK(zero_cpu_adam(g16, w, m, v, p16, n, 1, 1e-3f, 0.9f, 0.999f, 1e-8f, ZERO_MODE_STANDARD, 2) == ZERO_OK);
    for (int i = 0; i < n; ++i) {
        const float step = w[i] - 0.5f;
        CHECK(fabsf(fabsf(step) - 1e-3f) < 1e-6f);
        CHECK((step < 0.0f) == (i % 2 == 0));
    }
    CHECK(zero_cpu_adam(g16, w, m, v, p16, n, 0, 1e-3f, 0.9f, 0.999f, 1e-8f, 0, 2) == ZERO_EINVAL);

    CHECK(zero_strerror(ZERO_EOVERLAP) != NULL && zero_strerror(ZERO_EOVERLAP)[0] != '\0');
    puts("ok");
    return 0;
}
"""


def test_header_compiles_as_c11_and_host_entry_points_work(zlib, tmp_path):
    gcc = shutil.which("gcc")
    if gcc is None:
        pytest.skip("no C compiler")
    so = zlib._LIB_PATH
    src = tmp_path / "abi_check.c"
    src.write_text(C_PROGRAM)
    exe = tmp_path / "abi_check"
    cmd = [gcc, "-std=c11", "-Wall", "-Wextra", "-Werror", "-pedantic", "-I", os.path.join(ROOT, "include"),
           str(src), "-o", str(exe), so, f"-Wl,-rpath,{os.path.dirname(so)}", "-lm"]
    r = subprocess.run(cmd, capture_output=True, text=True)
    assert r.returncode == 0, r.stderr
    env = dict(os.environ)
    r = subprocess.run([str(exe)], capture_output=True, text=True, env=env, timeout=120)
    assert r.returncode == 0 and r.stdout.strip() == "ok", r.stderr + r.stdout
