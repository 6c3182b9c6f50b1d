"""The forward kernel's work schedule (csrc/fat_schedule.h), built for the host.

For every launch shape the host can choose, every query tile (item) must go
to exactly one block, each block's item sequence must end (the index grows
with k, so the first -1 is the last item), and no block may take more than
kMaxDeferred items: a block's list of tiles deferred to the fallback pass
holds that many, so a larger share would drop flagged tiles from the second
pass.  With one block per item, block b takes item b and nothing else.
"""
import os
import shutil
import subprocess

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
CSRC = os.path.join(ROOT, "tensorized_online_softmax_gb300", "csrc")

HARNESS = r"""
#include <cstdio>
#include <cstdlib>
#include <vector>
#include "fat_schedule.h"

// argv: n_items sms one_per_item; prints "grid max_items_per_block" or an error
int main(int argc, char** argv) {
  const int n = std::atoi(argv[1]), sms = std::atoi(argv[2]);
  const bool one = std::atoi(argv[3]) != 0;
  const int G = fat::fwd_grid(n, sms, one);
  if (G < 1 || G > n) { std::printf("bad grid %d\n", G); return 1; }
  std::vector<int> seen(n, 0);
  int most = 0;
  for (int b = 0; b < G; ++b) {
    int k = 0, last = -1;
    for (;; ++k) {
      const int idx = fat::fwd_item_index(k, b, G, n);
      if (idx < 0) break;
      if (idx <= last || idx >= n) { std::printf("block %d: item %d after %d\n", b, idx, last); return 1; }
      last = idx;
      ++seen[idx];
    }
    // past the end stays past the end
    for (int extra = 1; extra <= 3; ++extra)
      if (fat::fwd_item_index(k + extra, b, G, n) >= 0) { std::printf("block %d resumes\n", b); return 1; }
    if (one && (k != 1 || fat::fwd_item_index(0, b, G, n) != b)) { std::printf("block %d\n", b); return 1; }
    if (k > most) most = k;
  }
  for (int i = 0; i < n; ++i)
    if (seen[i] != 1) { std::printf("item %d taken %d times\n", i, seen[i]); return 1; }
  if (most > fat::kMaxDeferred) { std::printf("block takes %d items\n", most); return 1; }
  std::printf("%d %d\n", G, most);
  return 0;
}
"""


@pytest.fixture(scope="module")
def harness(tmp_path_factory):
    cxx = shutil.which("g++")
    if cxx is None:
        pytest.skip("g++ not found")
    d = tmp_path_factory.mktemp("sched")
    src = d / "sched.cpp"
    src.write_text(HARNESS)
    exe = d / "sched"
    subprocess.run([cxx, "-std=c++17", "-O1", "-I", CSRC, "-o", str(exe), str(src)], check=True)
    return str(exe)


def run(harness, n, sms, one):
    r = subprocess.run([harness, str(n), str(sms), str(int(one))], capture_output=True, text=True)
    assert r.returncode == 0, f"n={n} sms={sms} one={one}: {r.stdout}"
    grid, most = (int(x) for x in r.stdout.split())
    return grid, most


@pytest.mark.parametrize("sms", [1, 2, 148, 152, 160])
@pytest.mark.parametrize("n", [1, 5, 151, 152, 153, 300, 2048, 4095, 9728, 9729, 100000])
def test_every_tile_once_and_within_the_deferred_list(harness, n, sms):
    grid, most = run(harness, n, sms, False)
    if n <= sms:
        assert grid == n and most == 1
    else:
        assert grid >= sms
        # one wave of persistent blocks unless the deferred list forces more
        if n <= sms * 64:
            assert grid == sms
    g1, m1 = run(harness, n, sms, True)
    assert g1 == n and m1 == 1


def test_headline_shape_takes_thirteen_or_fourteen_tiles_per_block(harness):
    # B2 H16 N8192: 2048 query tiles over 152 SMs
    grid, most = run(harness, 2 * 16 * 64, 152, False)
    assert grid == 152 and most == 14
