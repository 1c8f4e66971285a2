"""The boundary used from C: a C99 program (compiled with -pedantic -Werror)
includes include/tpgqa.h, links libtpgqa.so and calls the host-side entry points
(plan, q->kv map, status strings, an empty linear call). Its plan must equal the
oracle's; the header must also compile as C++. No GPU is touched."""
import os
import shutil
import subprocess

import pytest

import oracle as O
import tensor_sharded_linear_gqa_gb300 as tp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
PKG = os.path.join(ROOT, "tensor_sharded_linear_gqa_gb300")

PROGRAM = r"""
#include "tpgqa.h"
#include <stdio.h>

int main(int argc, char **argv) {
  tp_dims d;
  tp_plan *plan = NULL;
  int32_t map[256];
  int r, j;
  if (argc != 7) return 2;
  if (sscanf(argv[1], "%d", &d.tp_size) != 1 || sscanf(argv[2], "%d", &d.hidden) != 1 ||
      sscanf(argv[3], "%d", &d.num_q_heads) != 1 || sscanf(argv[4], "%d", &d.num_kv_heads) != 1 ||
      sscanf(argv[5], "%d", &d.head_dim) != 1 || sscanf(argv[6], "%d", &d.ffn) != 1)
    return 2;
  printf("version %s\n", tp_version());
  printf("create %s\n", tp_status_str(tp_plan_create(&d, &plan)));
  if (!plan) return 0;
  for (r = 0; r < d.tp_size; ++r) {
    tp_rank_shard s;
    int nq;
    if (tp_plan_query_rank(plan, r, &s) != TP_OK) return 3;
    printf("rank %d q %d %d kv %d %d rep %d", r, s.q_head_begin, s.q_head_end, s.kv_head_begin,
           s.kv_head_end, s.kv_replicated);
    for (j = 0; j < TP_W_COUNT; ++j)
      printf(" w%d %d %d %lld %lld", j, s.strategy[j], s.comm[j], (long long)s.range_begin[j],
             (long long)s.range_end[j]);
    nq = s.q_head_end - s.q_head_begin;
    if (tp_plan_q_to_kv(plan, r, map, 256) != TP_OK) return 4;
    printf(" map");
    for (j = 0; j < nq; ++j) printf(" %d", map[j]);
    printf("\n");
  }
  {
    /* zero tokens: valid, enqueues nothing */
    tp_tensor x = {0}, w[1], y[1];
    x.dtype = TP_BF16; x.rows = 0; x.cols = 64; x.ld = 64;
    w[0] = x; w[0].rows = 32; w[0].ptr = (void *)(uintptr_t)4096;
    y[0] = x; y[0].cols = 32; y[0].ld = 32;
    printf("empty %s\n", tp_status_str(tp_column_linear(1, &x, w, y, 1, NULL)));
  }
  printf("destroy %s\n", tp_status_str(tp_plan_destroy(plan)));
  return 0;
}
"""

NAMES = ["q_proj", "k_proj", "v_proj", "o_proj", "gate_proj", "up_proj", "down_proj"]


@pytest.fixture(scope="module")
def program(tmp_path_factory):
    if not shutil.which("gcc"):
        pytest.skip("no C compiler")
    tp.load()  # builds nothing; fails loudly when the library is missing
    d = tmp_path_factory.mktemp("cabi")
    src = d / "prog.c"
    src.write_text(PROGRAM)
    exe = d / "prog"
    subprocess.run(["gcc", "-std=c99", "-Wall", "-Wextra", "-pedantic", "-Werror", "-I",
                    os.path.join(ROOT, "include"), str(src), "-L", PKG, "-ltpgqa", f"-Wl,-rpath,{PKG}", "-o",
                    str(exe)], check=True, capture_output=True, text=True)
    return str(exe)


def run(program, *dims):
    out = subprocess.run([program, *map(str, dims)], capture_output=True, text=True, timeout=60)
    assert out.returncode == 0, out.stderr
    return out.stdout.splitlines()


@pytest.mark.parametrize("dims", [(4, 4096, 32, 8, 128, 14336), (8, 4096, 32, 4, 128, 14336),
                                  (8, 8192, 64, 8, 128, 28672), (2, 2048, 16, 4, 128, 8192), (1, 512, 4, 4, 128, 64)])
def test_c_program_sees_the_oracle_plan(program, dims):
    lines = run(program, *dims)
    assert lines[0].startswith("version tpgqa")
    assert lines[1] == "create TP_OK"
    ref = O.shard_plan(*dims)
    rows = [ln.split() for ln in lines if ln.startswith("rank ")]
    assert len(rows) == dims[0]
    for s, f in zip(ref, rows):
        assert int(f[1]) == s.rank
        assert (int(f[3]), int(f[4])) == tuple(s.q_heads)
        assert (int(f[6]), int(f[7])) == tuple(s.kv_heads)
        assert int(f[9]) == int(s.kv_replicated)
        for j, name in enumerate(NAMES):
            k = 10 + 5 * j
            assert f[k] == f"w{j}"
            assert (int(f[k + 3]), int(f[k + 4])) == tuple(s.ranges[name]), name
        m = f.index("map")
        assert [int(v) for v in f[m + 1:]] == list(s.q_to_kv)
    assert lines[-2] == "empty TP_OK"
    assert lines[-1] == "destroy TP_OK"


def test_c_program_gets_the_gqa_error(program):
    lines = run(program, 8, 4096, 32, 12, 128, 14336)  # 12 kv heads over 8 ranks: neither rule applies
    assert lines[1] == "create TP_ERR_GQA_SHAPE"


def test_header_compiles_as_cpp(tmp_path):
    if not shutil.which("g++"):
        pytest.skip("no C++ compiler")
    src = tmp_path / "h.cpp"
    src.write_text('#include "tpgqa.h"\nint main() { return tp_version() ? 0 : 1; }\n')
    subprocess.run(["g++", "-std=c++17", "-Wall", "-Wextra", "-pedantic", "-Werror", "-I",
                    os.path.join(ROOT, "include"), str(src), "-L", PKG, "-ltpgqa", f"-Wl,-rpath,{PKG}", "-o",
                    str(tmp_path / "h")], check=True, capture_output=True, text=True)
    assert subprocess.run([str(tmp_path / "h")], timeout=60).returncode == 0
