"""The wide kernels' index arithmetic (csrc/rmsnorm_wide_layout.h), compiled
for the host and checked exhaustively over element sizes, row lengths, row
starts and operand offsets, without a GPU:

- the split of a row: the head reaches the first 16-byte boundary, the body
  is whole 16-byte vectors, the tail is shorter than a vector;
- another operand read in that frame: body vector v is exactly that operand's
  bytes for the vector's columns, and both aligned chunks it is built from lie
  in the operand row's enclosing 16-byte span (so no read leaves the 16-byte
  granules the row touches); the same for gamma's one or two chunks a vector;
- the head and tail elements go to distinct threads, each exactly once;
- the shared-memory partial row is a bijection of the columns into its size,
  with 16-byte aligned float4s for the body;
- the L2 request of a row covers it with 16-byte aligned bounds.
"""
import os
import shutil
import subprocess

import pytest

from tests.conftest import ROOT

CSRC = os.path.join(ROOT, "row_wise_normalization_02_gb300", "csrc")

PROGRAM = r"""
#include <stdio.h>
#include <stdint.h>
#include <vector>
#include "rmsnorm_wide_layout.h"
using namespace rmsn;

static int bad = 0;
#define CHECK(c, ...) do { if (!(c)) { if (bad < 20) { printf(__VA_ARGS__); printf("\n"); } ++bad; } } while (0)

static uintptr_t lo16(uintptr_t a) { return a & ~(uintptr_t)15; }
static uintptr_t hi16(uintptr_t a) { return (a + 15) & ~(uintptr_t)15; }

int main() {
  const int Ns[] = {1, 2, 3, 5, 7, 8, 9, 15, 16, 17, 31, 33, 64, 127, 129, 255, 256, 257,
                    1000, 1001, 1032, 2049, 4096, 4100, 8191, 12288, 20000, 20001};
  const int pairs[3][2] = {{4, 4}, {2, 2}, {2, 4}};   // (x, gamma) element sizes
  const int Ts[] = {64, 96, 256, 384, 512};
  for (const auto& pr : pairs) {
    const int es = pr[0], ws = pr[1], E = 16 / es, GW = E * ws / 16;
    for (int N : Ns) {
      const uint64_t rb = (uint64_t)N * es;
      for (int oy = 0; oy < 16; oy += es) {
        for (int r = 0; r < 3; ++r) {   // rows 0-2: the split moves when rb % 16 != 0
          const uintptr_t a = 4096 + oy + r * rb;
          const int head = wide_head(a, N, es), nv = wide_nv(N, head, es);
          CHECK(head >= 0 && head <= N, "head %d N %d", head, N);
          CHECK(head == N || ((a + (uintptr_t)head * es) & 15) == 0, "head not at a boundary");
          CHECK(head == N || head < E, "head %d >= E", head);
          const int t0 = head + nv * E;
          CHECK(t0 <= N && (head == N ? nv == 0 : N - t0 < E), "tail N %d t0 %d", N, t0);
          // head and tail elements: distinct threads, each once
          for (int T : Ts) {
            std::vector<int> seen(N, 0);
            for (int tid = 0; tid < T; ++tid) {
              const int j = wide_edge_elem(head, nv, E, N, tid, T);
              if (j < 0) continue;
              CHECK(j < N && (j < head || j >= t0), "edge %d of body", j);
              if (j >= 0 && j < N) seen[j]++;
            }
            for (int j = 0; j < N; ++j) {
              const bool edge = j < head || j >= t0;
              CHECK(seen[j] == (edge ? 1 : 0), "element %d taken %d times (T %d)", j, seen[j], T);
            }
          }
          // other operands (x, dy, h, dres) at every offset
          for (int ob = 0; ob < 16; ob += es) {
            const uintptr_t b = 65536 + ob + r * rb;
            const WideSrc s = wide_src(b, head, es);
            CHECK((s.base & 15) == 0 && s.s >= 0 && s.s < 16, "src");
            for (int v = 0; v < nv; ++v) {
              const uintptr_t want = b + (uintptr_t)(head + v * E) * es;
              CHECK(s.base + 16 * (uintptr_t)v + s.s == want, "vector %d bytes", v);
              const uintptr_t c0 = s.base + 16 * (uintptr_t)v, c1 = c0 + 16;
              CHECK(c0 >= lo16(b) && c0 + 16 <= hi16(b + rb), "chunk 0 of %d out of span", v);
              if (s.s) CHECK(c1 >= lo16(b) && c1 + 16 <= hi16(b + rb), "chunk 1 of %d out of span", v);
            }
          }
          // gamma at every offset: GW chunks a vector, one more when shifted
          for (int og = 0; og < 16; og += ws) {
            const uintptr_t g = 131072 + og;
            const WideSrc s = wide_src(g, head, ws);
            for (int v = 0; v < nv; ++v) {
              CHECK(s.base + 16 * (uintptr_t)GW * v + s.s == g + (uintptr_t)(head + v * E) * ws,
                    "gamma vector %d", v);
              for (int k = 0; k < GW + (s.s ? 1 : 0); ++k) {
                const uintptr_t c = s.base + 16 * (uintptr_t)(GW * v + k);
                CHECK(c >= lo16(g) && c + 16 <= hi16(g + (uint64_t)N * ws), "gamma chunk");
              }
            }
          }
          // the L2 request of the row
          const uintptr_t l = wide_l2_lo(a);
          const uint32_t n = wide_l2_bytes(a, rb);
          CHECK(l % 16 == 0 && n % 16 == 0 && l <= a && l + n >= a + rb && n < rb + 32, "l2");
        }
        // the backward's partial row (rows a multiple of 16 bytes)
        if (rb % 16 == 0) {
          const uintptr_t a = 4096 + oy;
          const int head = wide_head(a, N, es), nv = wide_nv(N, head, es);
          const int F = wide_acc_floats(N, E);
          std::vector<int> hit(F, 0);
          for (int j = 0; j < N; ++j) {
            const int i = wide_acc_col(j, head, nv, E);
            CHECK(i >= 0 && i < F, "column %d at %d of %d", j, i, F);
            if (i >= 0 && i < F) hit[i]++;
          }
          for (int i = 0; i < F; ++i) CHECK(hit[i] <= 1, "offset %d used twice", i);
          for (int v = 0; v < nv; ++v)
            for (int w = 0; w < E / 4; ++w) {
              const int o = wide_acc_vec(v, w, E);
              CHECK(o % 4 == 0 && o + 4 <= F, "float4 %d,%d", v, w);
              for (int k = 0; k < 4; ++k)
                CHECK(wide_acc_col(head + v * E + 4 * w + k, head, nv, E) == o + k, "vec/col");
            }
        }
      }
    }
  }
  // rows beyond 16 MB are not requested
  CHECK(wide_l2_bytes(16, (uint64_t)1 << 25) == 0, "l2 cap");
  printf(bad ? "FAIL %d\n" : "PASS\n", bad);
  return bad ? 1 : 0;
}
"""


def test_wide_layout_index_arithmetic(tmp_path):
    cxx = shutil.which("g++")
    if cxx is None:
        pytest.skip("no host C++ compiler")
    src = tmp_path / "layout.cpp"
    src.write_text(PROGRAM)
    exe = tmp_path / "layout"
    r = subprocess.run([cxx, "-std=c++17", "-O1", "-Wall", "-Werror", "-I", CSRC, str(src), "-o",
                        str(exe)], capture_output=True, text=True)
    assert r.returncode == 0, r.stderr
    out = subprocess.run([str(exe)], capture_output=True, text=True, timeout=300)
    assert out.returncode == 0 and "PASS" in out.stdout, out.stdout + out.stderr
