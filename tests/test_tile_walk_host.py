"""Host test of the tile walk the tensor-core kernels share (csrc/common.cuh,
TileWalk): the jumps of the query-stationary walks (forward, dQ) over the key
tiles the causal mask hides, and of the key-stationary walk (the dK/dV kernel's
producer) over the query tiles that cannot see its key tile, visit exactly the
tiles, in exactly the order, that stepping through every tile and skipping the
hidden ones one by one visits.  Both layouts, several cp, chunk sizes, passes,
first chunks and directions, every anchor tile.

The struct is compiled from the header itself with the host compiler (its device
qualifiers defined away), so the test checks the code the kernels use."""
import os
import re
import shutil
import subprocess

import pytest

from conftest import ROOT

HEADER = os.path.join(ROOT, "blockwise_online_softmax_cpattn_gb300", "csrc", "common.cuh")

DRIVER = r"""
#include <cstdio>
#include <vector>
#define __device__
#define __host__
#define __forceinline__ inline
%STRUCTS%
// reference: every tile in turn, hidden ones skipped one at a time
// (a key tile is hidden from the query tile at q0 when it starts past q0 + 127)
static std::vector<int> plain(const SeqMap& m, int first, int n, int dir, int reps, int q0) {
  std::vector<int> out;
  TileWalk w;
  for (w.start(m, first, n, dir, reps); !w.done(); w.next())
    if (!(w.pos() > q0 + 127)) out.push_back(w.i * 1000000 + w.rep * 10000 + w.slot() / 128);
  return out;
}
static std::vector<int> jumped(const SeqMap& m, int first, int n, int dir, int reps, int q0) {
  std::vector<int> out;
  TileWalk w;
  w.start(m, first, n, dir, reps);
  w.settle_keys(q0);
  while (!w.done()) {
    out.push_back(w.i * 1000000 + w.rep * 10000 + w.slot() / 128);
    w.next();
    w.settle_keys(q0);
  }
  return out;
}
// key-stationary: a query tile at qpos is hidden from the key tile at k0 when k0 is
// past qpos + 127
static std::vector<int> plain_q(const SeqMap& m, int first, int n, int dir, int reps, int k0) {
  std::vector<int> out;
  TileWalk w;
  for (w.start(m, first, n, dir, reps); !w.done(); w.next())
    if (!(k0 > w.pos() + 127)) out.push_back(w.i * 1000000 + w.rep * 10000 + w.slot() / 128);
  return out;
}
static std::vector<int> jumped_q(const SeqMap& m, int first, int n, int dir, int reps, int k0) {
  std::vector<int> out;
  TileWalk w;
  w.start(m, first, n, dir, reps);
  w.settle_queries(k0);
  while (!w.done()) {
    out.push_back(w.i * 1000000 + w.rep * 10000 + w.slot() / 128);
    w.next();
    w.settle_queries(k0);
  }
  return out;
}
int main() {
  long cases = 0, bad = 0;
  const int cps[] = {1, 2, 3, 4, 5, 8};
  for (int zz = 0; zz < 2; ++zz)
    for (int cp : cps)
      for (int mult = 1; mult <= 3; ++mult) {
        const int c = (zz ? 256 : 128) * mult;
        const SeqMap m = SeqMap::make(cp * c, cp, zz);
        for (int reps : {1, 2, 4})
          for (int first = 0; first < cp; ++first)
            for (int n : {1, cp})
              for (int dir : {-1, 1})
                for (int q0 = 0; q0 < m.T; q0 += 128) {
                  ++cases;
                  if (plain(m, first, n, dir, reps, q0) != jumped(m, first, n, dir, reps, q0) &&
                      ++bad < 5)
                    std::printf("mismatch zz=%d cp=%d c=%d reps=%d first=%d n=%d dir=%d q0=%d\n",
                                zz, cp, c, reps, first, n, dir, q0);
                  ++cases;  // the same anchor as a key tile of the key-stationary walk
                  if (plain_q(m, first, n, dir, reps, q0) != jumped_q(m, first, n, dir, reps, q0) &&
                      ++bad < 5)
                    std::printf("mismatch (queries) zz=%d cp=%d c=%d reps=%d first=%d n=%d "
                                "dir=%d k0=%d\n", zz, cp, c, reps, first, n, dir, q0);
                }
      }
  std::printf("cases %ld mismatches %ld\n", cases, bad);
  return bad != 0;
}
"""


def _struct(src, name):
    m = re.search(r"^struct %s \{.*?^\};" % name, src, re.S | re.M)
    assert m, name
    return m.group(0)


def test_tile_walk_jumps_visit_the_same_tiles(tmp_path):
    gxx = shutil.which("g++")
    if gxx is None:
        pytest.skip("no host C++ compiler")
    src = open(HEADER).read()
    code = DRIVER.replace("%STRUCTS%", _struct(src, "SeqMap") + "\n" + _struct(src, "TileWalk"))
    cpp = tmp_path / "walk.cpp"
    cpp.write_text(code)
    exe = tmp_path / "walk"
    subprocess.run([gxx, "-O1", "-std=c++17", str(cpp), "-o", str(exe)], check=True,
                   capture_output=True, text=True)
    r = subprocess.run([str(exe)], capture_output=True, text=True, timeout=120)
    assert r.returncode == 0, r.stdout
    assert "mismatches 0" in r.stdout and "cases 0 " not in r.stdout
