"""The C oracle under AddressSanitizer and UndefinedBehaviorSanitizer (host
only): a small driver runs attention, block mass and the aggregation on a
tiny ragged case in all three element modes; any sanitizer report fails."""
import shutil
import subprocess
from pathlib import Path

import pytest

ORACLE_C = Path(__file__).resolve().parents[1] / "oracle" / "kvs_oracle.c"

DRIVER = r"""
#include <stdint.h>
#include <stdio.h>
#include <stdlib.h>
int orc_decode_heads(const uint16_t *, const uint16_t *, const uint16_t *, int64_t, int, int, int,
                     int, int, const int32_t *, int, int, double *, double *, double *);
int orc_decode_heads_u8(const uint16_t *, const uint8_t *, const uint8_t *, const double *,
                        const double *, int64_t, int, int, int, int, int, const int32_t *, int, int,
                        double *, double *, double *);
int orc_decode_heads_f32(const uint16_t *, const float *, const float *, int64_t, int, int, int,
                         int, int, const int32_t *, int, int, double *, double *, double *);
void orc_aggregate_mass(const double *, int64_t, int, int, int, double *);
int main(void) {
    const int L = 2, Hq = 8, Hkv = 2, d = 64, B = 16;
    const int64_t n = 37;                       /* ragged: 3 blocks, the last partial */
    const int nb = (int)((n + B - 1) / B), nh = L * Hq;
    uint16_t *q = malloc(sizeof(uint16_t) * L * Hq * d);
    uint16_t *k = malloc(sizeof(uint16_t) * n * L * Hkv * d), *v = malloc(sizeof(uint16_t) * n * L * Hkv * d);
    uint8_t *k8 = malloc(n * L * Hkv * d), *v8 = malloc(n * L * Hkv * d);
    float *kf = malloc(sizeof(float) * n * L * Hkv * d), *vf = malloc(sizeof(float) * n * L * Hkv * d);
    double lut[256], *out = malloc(sizeof(double) * nh * d), *lse = malloc(sizeof(double) * nh);
    double *hm = malloc(sizeof(double) * nh * nb), *mass = malloc(sizeof(double) * nb);
    uint32_t s = 12345;
    for (int i = 0; i < L * Hq * d; ++i) { s = s * 1664525u + 1013904223u; q[i] = (uint16_t)(0x3c00 + (s >> 24)); }
    for (int64_t i = 0; i < n * L * Hkv * d; ++i) {
        s = s * 1664525u + 1013904223u;
        k[i] = (uint16_t)(0x3c00 + (s >> 25)); v[i] = (uint16_t)(0xbc00 + (s >> 26));
        k8[i] = (uint8_t)(s >> 8); v8[i] = (uint8_t)(s >> 16);
        kf[i] = (float)(s >> 20) / 4096.0f - 0.5f; vf[i] = (float)(s >> 12 & 0xff) / 256.0f;
    }
    for (int i = 0; i < 256; ++i) lut[i] = (i - 128) / 64.0;
    int rc = 0;
    for (int threads = 1; threads <= 3; threads += 2) {
        rc |= orc_decode_heads(q, k, v, n, L, Hq, Hkv, d, B, NULL, nh, threads, out, lse, hm);
        rc |= orc_decode_heads_u8(q, k8, v8, lut, lut, n, L, Hq, Hkv, d, B, NULL, nh, threads, out, lse, hm);
        rc |= orc_decode_heads_f32(q, kf, vf, n, L, Hq, Hkv, d, B, NULL, nh, threads, out, lse, hm);
    }
    orc_aggregate_mass(hm, nb, L, Hq, Hkv, mass);
    double total = 0;
    for (int b = 0; b < nb; ++b) total += mass[b];
    printf("rc=%d mass_sum=%.12f\n", rc, total);
    free(q); free(k); free(v); free(k8); free(v8); free(kf); free(vf);
    free(out); free(lse); free(hm); free(mass);
    return rc != 0 || total < 0.999999 || total > 1.000001;
}
"""


@pytest.mark.skipif(shutil.which("gcc") is None, reason="needs gcc")
def test_oracle_clean_under_asan_ubsan(tmp_path):
    drv = tmp_path / "drv.c"
    drv.write_text(DRIVER)
    exe = tmp_path / "drv"
    flags = ["-O1", "-g", "-fsanitize=address,undefined", "-fno-sanitize-recover=all",
             "-fno-omit-frame-pointer", "-pthread"]
    r = subprocess.run(["gcc", *flags, str(drv), str(ORACLE_C), "-o", str(exe), "-lm"],
                       capture_output=True, text=True)
    if r.returncode != 0 and "sanitizer" in (r.stderr + r.stdout).lower():
        pytest.skip("sanitizer runtime not available: " + r.stderr[-200:])
    assert r.returncode == 0, r.stderr
    run = subprocess.run([str(exe)], capture_output=True, text=True,
                         env={"ASAN_OPTIONS": "detect_leaks=1", "UBSAN_OPTIONS": "print_stacktrace=1"})
    assert run.returncode == 0, run.stdout + run.stderr
    assert "ERROR" not in run.stderr and "runtime error" not in run.stderr, run.stderr
    assert "rc=0" in run.stdout
