"""The kernels' work schedules (csrc/fat_schedule.h), built for the host.

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


BWD_HARNESS = r"""
#include <cstdio>
#include <cstdlib>
#include <vector>
#include "fat_schedule.h"

// argv: BH n_blocks causal max_heads; prints "groups group_heads group_extra"
// after checking that CTA -> (jb, bh) is a bijection, that a group's heads are
// consecutive, at most max_heads and within one of each other, and that the
// key blocks of a group come in order (the heaviest causal ones first)
int main(int argc, char** argv) {
  const int BH = std::atoi(argv[1]), nb = std::atoi(argv[2]);
  const bool causal = std::atoi(argv[3]) != 0;
  const int cap = std::atoi(argv[4]);
  const int gh = fat::bwd_group_heads(BH, cap), ge = fat::bwd_group_extra(BH, cap);
  const int ng = fat::bwd_group_count(BH, cap);
  if (gh * ng + ge != BH || ge >= ng || gh < 1 || gh + (ge > 0) > cap) {
    std::printf("bad groups %d %d %d\n", ng, gh, ge); return 1;
  }
  std::vector<int> seen(static_cast<size_t>(BH) * nb, 0);
  int prev_jb = -1, prev_head0 = -1;
  for (int idx = 0; idx < BH * nb; ++idx) {
    int jb, bh;
    fat::bwd_work_item(idx, nb, causal, gh, ge, jb, bh);
    if (jb < 0 || jb >= nb || bh < 0 || bh >= BH) { std::printf("idx %d out of range\n", idx); return 1; }
    ++seen[static_cast<size_t>(bh) * nb + jb];
    if (causal) {
      // group of this CTA: the first ge groups have gh + 1 heads
      const int big = (gh + 1) * nb;
      const int g = idx < ge * big ? idx / big : ge + (idx - ge * big) / (gh * nb);
      const int size = g < ge ? gh + 1 : gh;
      const int head0 = g < ge ? g * (gh + 1) : ge * (gh + 1) + (g - ge) * gh;
      if (bh < head0 || bh >= head0 + size) { std::printf("idx %d head %d outside its group\n", idx, bh); return 1; }
      if (head0 != prev_head0) { prev_head0 = head0; prev_jb = -1; }
      if (jb < prev_jb) { std::printf("idx %d: key block %d after %d\n", idx, jb, prev_jb); return 1; }
      prev_jb = jb;
    } else if (jb != idx % nb || bh != idx / nb) {
      std::printf("idx %d not head-major\n", idx); return 1;
    }
  }
  for (size_t i = 0; i < seen.size(); ++i)
    if (seen[i] != 1) { std::printf("(jb, bh) %zu taken %d times\n", i, seen[i]); return 1; }
  std::printf("%d %d %d\n", ng, gh, ge);
  return 0;
}
"""


@pytest.fixture(scope="module")
def bwd_harness(tmp_path_factory):
    cxx = shutil.which("g++")
    if cxx is None:
        pytest.skip("g++ not found")
    d = tmp_path_factory.mktemp("bwdsched")
    src = d / "bwd.cpp"
    src.write_text(BWD_HARNESS)
    exe = d / "bwd"
    subprocess.run([cxx, "-std=c++17", "-O1", "-I", CSRC, "-o", str(exe), str(src)], check=True)
    return str(exe)


def run_bwd(harness, BH, nb, causal, cap):
    r = subprocess.run([harness, str(BH), str(nb), str(int(causal)), str(cap)],
                       capture_output=True, text=True)
    assert r.returncode == 0, f"BH={BH} nb={nb} causal={causal} cap={cap}: {r.stdout}"
    return tuple(int(x) for x in r.stdout.split())


@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("BH,nb,cap", [(1, 1, 1), (1, 3, 8), (7, 2, 3), (32, 64, 6), (64, 16, 24),
                                       (32, 128, 12), (5, 9, 5), (13, 4, 1), (100, 3, 7)])
def test_backward_blocks_each_once_in_balanced_groups(bwd_harness, BH, nb, causal, cap):
    run_bwd(bwd_harness, BH, nb, causal, cap)


def test_headline_backward_groups_are_six_six_five_five_five_five(bwd_harness):
    # B2 H16 N8192 d128 causal: Q, dO, dQ of 6 heads fill the 48 MiB L2 share,
    # so 32 heads run as 6 groups, two of 6 heads and four of 5 (not 6 x 5 + 2)
    assert run_bwd(bwd_harness, 32, 64, True, 6) == (6, 5, 2)
