"""Memory safety of the library's host C++ (the layout table, the bucket
planner and the host Adam with its thread pool): the two sources are built
with AddressSanitizer and UndefinedBehaviorSanitizer together with a C driver
that calls them on seeded random inputs -- tensor lists with empty tensors,
every stage, rank counts up to ZERO_MAX_RANKS, the two-call bucket pattern,
host Adam on ragged lengths from four threads at once -- and checks a few
invariants on the way.  Any out-of-bounds access, leak or undefined
operation makes the program fail.  No CUDA is involved."""
import os
import shutil
import subprocess

import pytest

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(HERE)
CSRC = os.path.join(ROOT, "zero_sharded_mixed_shard_gb300", "csrc")

DRIVER = r"""
#include <pthread.h>
#include <stdio.h>
#include <stdlib.h>
#include <string.h>

#include "zero_step.h"

#define CHECK(cond)                                                \
    do {                                                           \
        if (!(cond)) {                                             \
            fprintf(stderr, "line %d: %s\n", __LINE__, #cond);     \
            exit(1);                                               \
        }                                                          \
    } while (0)

static unsigned long long rnd_r(unsigned long long* state)   /* splitmix64 */
{
    unsigned long long z = (*state += 0x9E3779B97F4A7C15ull);
    z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9ull;
    z = (z ^ (z >> 27)) * 0x94D049BB133111EBull;
    return z ^ (z >> 31);
}
static unsigned long long main_state = 1;
static unsigned long long rnd(void) { return rnd_r(&main_state); }

static void layouts(void)
{
    for (int iter = 0; iter < 300; ++iter) {
        int nt = 1 + (int)(rnd() % 40);
        int64_t numel[40];
        int64_t total = 0;
        for (int i = 0; i < nt; ++i) {
            numel[i] = (rnd() % 4 == 0) ? 0 : (int64_t)(rnd() % 5000);
            total += numel[i];
        }
        if (total == 0) numel[0] = total = 1;
        int32_t P = 1 + (int32_t)(rnd() % (iter % 3 == 0 ? ZERO_MAX_RANKS : 70));
        int32_t stage = (int32_t)(rnd() % 4);
        zero_layout_t L;
        memset(&L, 0, sizeof L);
        CHECK(zero_init_layout(numel, nt, P, stage, &L) == ZERO_OK);
        int64_t covered = 0;
        for (int32_t k = 0; k < P; ++k) {
            int64_t b = -1, e = -1;
            CHECK(zero_shard_range(L.N, P, k, &b, &e) == ZERO_OK);
            CHECK(b == L.shard_begin[k] && e == L.shard_end[k]);
            for (int64_t s = L.seg_offsets[k]; s < L.seg_offsets[k + 1]; ++s) covered += L.segs[s].len;
        }
        CHECK(covered == total);
        zero_free_layout(&L);
        zero_free_layout(&L);

        int32_t nb = 0;
        int64_t be = 1 + (int64_t)(rnd() % 9000);
        int32_t backward = (int32_t)(rnd() % 2);
        CHECK(zero_plan_buckets(numel, nt, be, backward, NULL, 0, &nb) == ZERO_OK);
        CHECK(nb >= 1);
        zero_bucket_t* bk = (zero_bucket_t*)malloc(sizeof(zero_bucket_t) * (size_t)nb);
        CHECK(bk != NULL);
        CHECK(zero_plan_buckets(numel, nt, be, backward, bk, nb - 1, &nb) == ZERO_EINVAL || nb == 1);
        CHECK(zero_plan_buckets(numel, nt, be, backward, bk, nb, &nb) == ZERO_OK);
        int64_t sum = 0;
        for (int32_t b = 0; b < nb; ++b) sum += bk[b].end - bk[b].begin;
        CHECK(sum == total);
        free(bk);
        double bytes = 0, floats = 0, comm = 0;
        CHECK(zero_memory_bytes(total, P, stage, &bytes, &floats, &comm) == ZERO_OK);
    }
}

struct job {
    int id;
};

static void* adam_thread(void* arg)
{
    const int id = ((struct job*)arg)->id;
    unsigned long long state = 1000 + (unsigned long long)id;   /* one generator per thread */
    for (int iter = 0; iter < 12; ++iter) {
        int64_t n = 1 + (int64_t)(rnd_r(&state) % 70000);
        uint16_t* g = (uint16_t*)malloc((size_t)n * 2);
        uint16_t* p = (uint16_t*)malloc((size_t)n * 2);
        float* w = (float*)malloc((size_t)n * 4);
        float* m = (float*)malloc((size_t)n * 4);
        float* v = (float*)malloc((size_t)n * 4);
        CHECK(g && p && w && m && v);
        for (int64_t i = 0; i < n; ++i) {
            g[i] = (uint16_t)(rnd_r(&state) & 0xFFFF);   /* every fp16 code, inf and NaN included */
            w[i] = 0.01f * (float)(i % 97);
            m[i] = 0.0f;
            v[i] = 0.0f;
        }
        const int32_t threads = (int32_t)((id + iter) % 6);
        CHECK(zero_cpu_adam(g, w, m, v, p, n, 1 + iter, 1e-3f, 0.9f, 0.999f, 1e-8f, iter % 3, threads) == ZERO_OK);
        free(g); free(p); free(w); free(m); free(v);
    }
    return NULL;
}

int main(void)
{
    layouts();
    pthread_t th[4];
    struct job jobs[4];
    for (int i = 0; i < 4; ++i) {
        jobs[i].id = i;
        CHECK(pthread_create(&th[i], NULL, adam_thread, &jobs[i]) == 0);
    }
    for (int i = 0; i < 4; ++i) pthread_join(th[i], NULL);
    puts("ok");
    return 0;
}
"""


def test_host_code_under_address_and_ub_sanitizers(tmp_path):
    gxx, gcc = shutil.which("g++"), shutil.which("gcc")
    if gxx is None or gcc is None:
        pytest.skip("no C/C++ compiler")
    san = ["-fsanitize=address,undefined", "-fno-sanitize-recover=undefined", "-fno-omit-frame-pointer", "-g",
           "-O1"]
    inc = ["-I", os.path.join(ROOT, "include")]
    objs = []
    for src in ("layout.cpp", "cpu_adam.cpp"):
        obj = tmp_path / (src + ".o")
        r = subprocess.run([gxx, "-std=c++17", "-ffp-contract=off", "-pthread", *san, *inc, "-c",
                            os.path.join(CSRC, src), "-o", str(obj)], capture_output=True, text=True)
        if r.returncode != 0 and "sanitize" in r.stderr:
            pytest.skip("the compiler has no sanitizer runtime here")
        assert r.returncode == 0, r.stderr
        objs.append(str(obj))
    drv = tmp_path / "driver.c"
    drv.write_text(DRIVER)
    exe = tmp_path / "driver"
    r = subprocess.run([gcc, "-std=c11", *san, *inc, "-c", str(drv), "-o", str(tmp_path / "driver.o")],
                       capture_output=True, text=True)
    assert r.returncode == 0, r.stderr
    r = subprocess.run([gxx, *san, "-pthread", str(tmp_path / "driver.o"), *objs, "-o", str(exe)],
                       capture_output=True, text=True)
    if r.returncode != 0 and ("asan" in r.stderr or "ubsan" in r.stderr):
        pytest.skip("no sanitizer runtime to link against")
    assert r.returncode == 0, r.stderr
    env = dict(os.environ, ASAN_OPTIONS="detect_leaks=1:abort_on_error=0", UBSAN_OPTIONS="print_stacktrace=1")
    r = subprocess.run([str(exe)], capture_output=True, text=True, env=env, timeout=600)
    assert r.returncode == 0 and r.stdout.strip() == "ok", (r.stdout + r.stderr)[-4000:]
