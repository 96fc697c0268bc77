"""The device split planner (csrc/plan_device.cuh) run on the CPU.

`build_plan` is written for a group of NTHREADS GPU threads that meet at a
barrier and exchange values with warp shuffles.  Here the header itself is
compiled with g++ next to a stand-in for its device helpers: each GPU thread
is a host thread, the group barrier a std::barrier, a warp shuffle an
exchange through a 32-slot array between two barriers of the warp's 32
threads.  Its outputs (validated lengths, page prefix, first split, slot
bases, {G_eff, P}, the status word) are compared with the plan arithmetic
restated in test_plan_model.py, for the group sizes the kernels use (128
threads in the GEMM epilogue, 1024 in the plan and small-projection
kernels), batches larger than the group (the scan's carry across passes),
and lengths that need clamping (reported, detail 1000000 + first bad b).
"""
import os
import shutil
import subprocess

import numpy as np
import pytest

from test_plan_model import plan as model_plan

ROOT = os.path.join(os.path.dirname(__file__), "..")
CSRC = os.path.join(ROOT, "mla_latent_kv_82_b300", "csrc")
INCLUDE = os.path.join(ROOT, "include")
MLA_ERR_DEVICE_INDEX = 6

# Stand-in for device_util.cuh: only what plan_device.cuh uses.
HELPERS = r"""
#pragma once
#include <algorithm>
#include <atomic>
#include <barrier>
#include <cstdint>
#include "mla.h"
#define __device__
#define __forceinline__ inline
namespace mla {
using std::min;
struct WarpLink { std::barrier<>* bar; int* slots; };
inline thread_local WarpLink* t_warp = nullptr;
inline thread_local int t_lane = 0;
inline int __shfl_up_sync(unsigned, int x, int o) {
  t_warp->slots[t_lane] = x;
  t_warp->bar->arrive_and_wait();
  const int y = t_lane >= o ? t_warp->slots[t_lane - o] : x;
  t_warp->bar->arrive_and_wait();
  return y;
}
inline void __threadfence_block() { std::atomic_thread_fence(std::memory_order_seq_cst); }
// status = {code, detail, count}: the first report wins, later ones count
inline void report(int* status, int code, int detail) {
  int zero = 0;
  if (__atomic_compare_exchange_n(&status[0], &zero, code, false, __ATOMIC_SEQ_CST,
                                  __ATOMIC_SEQ_CST))
    __atomic_store_n(&status[1], detail, __ATOMIC_SEQ_CST);
  __atomic_fetch_add(&status[2], 1, __ATOMIC_SEQ_CST);
}
}  // namespace mla
"""

RUNNER = r"""
#include <cstdio>
#include <thread>
#include <vector>
#include "device_util.cuh"
#include "plan_device.cuh"
using namespace mla;

template <int N>
void run(PlanArgs a) {
  std::barrier<> group(N);
  std::vector<std::barrier<>*> warp_bars;
  std::vector<std::vector<int>> slots(N / 32, std::vector<int>(32));
  std::vector<WarpLink> links;
  for (int w = 0; w < N / 32; ++w) warp_bars.push_back(new std::barrier<>(32));
  for (int w = 0; w < N / 32; ++w) links.push_back({warp_bars[w], slots[w].data()});
  int tmp[33];
  std::vector<std::thread> th;
  for (int tid = 0; tid < N; ++tid)
    th.emplace_back([&, tid] {
      t_warp = &links[tid / 32];
      t_lane = tid % 32;
      build_plan<N>(tid, [&] { group.arrive_and_wait(); }, tmp, a);
    });
  for (auto& t : th) t.join();
  for (auto* b : warp_bars) delete b;
}

int main() {
  int n_cases;
  if (scanf("%d", &n_cases) != 1) return 1;
  for (int k = 0; k < n_cases; ++k) {
    int N, B, T, page, max_pages, max_position, G_max;
    if (scanf("%d %d %d %d %d %d %d", &N, &B, &T, &page, &max_pages, &max_position, &G_max) != 7)
      return 1;
    std::vector<int32_t> seq(B);
    for (auto& s : seq) if (scanf("%d", &s) != 1) return 1;
    std::vector<int> lens(B, -7), prefix(B + 1, -7), first(B, -7), slot_base(B + 1, -7),
        meta(4, -7), status(4, 0);
    PlanArgs a{seq.data(), B, T, page, max_pages, max_position, G_max, lens.data(),
               prefix.data(), first.data(), slot_base.data(), meta.data(), status.data()};
    if (N == 128) run<128>(a); else if (N == 1024) run<1024>(a); else return 2;
    auto put = [](const char* name, const std::vector<int>& v) {
      printf("%s", name);
      for (int x : v) printf(" %d", x);
      printf("\n");
    };
    put("lens", lens); put("prefix", prefix); put("first", first); put("slot_base", slot_base);
    put("meta", meta); put("status", status);
  }
  return 0;
}
"""


@pytest.fixture(scope="module")
def runner(tmp_path_factory):
    gxx = shutil.which("g++")
    if gxx is None:
        pytest.skip("needs g++")
    d = tmp_path_factory.mktemp("plan_device")
    # the real header, next to the stand-in for its helpers
    shutil.copy(os.path.join(CSRC, "plan_device.cuh"), d / "plan_device.cuh")
    (d / "device_util.cuh").write_text(HELPERS)
    (d / "runner.cpp").write_text(RUNNER)
    exe = d / "runner"
    subprocess.run([gxx, "-std=c++20", "-O1", "-pthread", "-I", str(d), "-I", INCLUDE,
                    str(d / "runner.cpp"), "-o", str(exe)], check=True)

    def run(cases):
        lines = [str(len(cases))]
        for c in cases:
            lines.append(" ".join(str(x) for x in
                                  (c["N"], len(c["seq"]), c["T"], c["page"], c["max_pages"],
                                   c["max_position"], c["G_max"])))
            lines.append(" ".join(str(x) for x in c["seq"]))
        out = subprocess.run([str(exe)], input="\n".join(lines) + "\n", check=True,
                             capture_output=True, text=True, timeout=300).stdout.splitlines()
        res = []
        for i in range(len(cases)):
            block = out[6 * i:6 * i + 6]
            res.append({ln.split()[0]: [int(x) for x in ln.split()[1:]] for ln in block})
        return res
    return run


def expected(c):
    cap = min(c["max_pages"] * c["page"], c["max_position"])
    lens = [min(max(s, c["T"]), cap) for s in c["seq"]]
    prefix, P, G, first, slot_base = model_plan(lens, c["page"], c["G_max"])
    bad = [b for b, (s, L) in enumerate(zip(c["seq"], lens)) if s != L]
    return {"lens": lens, "prefix": [int(x) for x in prefix], "first": [int(x) for x in first],
            "slot_base": [int(x) for x in slot_base], "meta": [G, P], "bad": bad}


def check(c, got):
    e = expected(c)
    for k in ("lens", "prefix", "first", "slot_base"):
        assert got[k] == e[k], (k, c)
    assert got["meta"][:2] == e["meta"], c
    code, detail, count = got["status"][:3]
    if e["bad"]:
        # threads report in any order: some bad b's report wins, every one counts
        assert code == MLA_ERR_DEVICE_INDEX and detail - 1000000 in e["bad"]
        assert count == len(e["bad"])
    else:
        assert (code, count) == (0, 0)


def _case(rng, N, B):
    page = 64
    max_pages = int(rng.integers(1, 200))
    T = int(rng.integers(1, 9))
    return {"N": N, "T": T, "page": page, "max_pages": max_pages,
            "max_position": int(rng.integers(T, 2 * max_pages * page + 2)),
            "G_max": int(rng.integers(1, 300)),
            "seq": [int(x) for x in rng.integers(0, max_pages * page + 100, B)]}


def test_group_of_128_matches_the_model(runner):
    rng = np.random.default_rng(11)
    cases = [_case(rng, 128, int(rng.integers(1, 400))) for _ in range(40)]
    for c, got in zip(cases, runner(cases)):
        check(c, got)


def test_group_of_1024_matches_the_model(runner):
    rng = np.random.default_rng(12)
    cases = [_case(rng, 1024, B) for B in (1, 5, 1023, 1024, 1025, 2500)]
    for c, got in zip(cases, runner(cases)):
        check(c, got)


def test_valid_lengths_report_nothing(runner):
    """Lengths inside [T, cap] pass unchanged and the status word stays 0;
    one page per split when the pages are few."""
    c = {"N": 128, "T": 2, "page": 64, "max_pages": 64, "max_position": 1 << 20, "G_max": 74,
         "seq": [2, 64, 65, 4096, 130]}
    got = runner([c])[0]
    check(c, got)
    assert got["status"][:3] == [0, 0, 0]
    assert got["meta"][:2] == [min(74, max(1, got["prefix"][-1] // 2)), got["prefix"][-1]]


def test_planted_slip_in_the_model_is_caught(runner):
    """The comparison is not vacuous: a model that forgot the clamp to
    max_position disagrees with the device code on such a case."""
    c = {"N": 128, "T": 1, "page": 64, "max_pages": 10, "max_position": 100, "G_max": 8,
         "seq": [300, 50]}
    got = runner([c])[0]
    check(c, got)
    wrong = [min(max(s, 1), 10 * 64) for s in c["seq"]]
    assert got["lens"] != wrong
