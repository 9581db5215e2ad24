"""Host logic of the paged KV cache's page pool (csrc/page_pool.h), compiled
with g++ and driven through scripted scenarios on the CPU: pages are handed
out in order as slots grow, no physical page backs two live entries (except
the training forward's explicit sharing), the scratch page is never handed
out and backs every other entry, exhaustion is reported, and a reset returns
everything."""
import os
import subprocess

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
CSRC = os.path.join(ROOT, "block_diffusion_speculative_ctx_gb300", "csrc")

DRIVER = r"""
#include <cstdio>
#include <cstring>
#include "page_pool.h"
using dfl::PagePool;
static PagePool P;
static void dump() {
    printf("T");
    for (int x : P.table()) printf(" %d", x);
    printf("\nU %d %d %d\nD %d", P.in_use(), P.capacity(), P.scratch(), P.full_dirty() ? 1 : 0);
    for (int e : P.pending()) printf(" %d", e);
    printf("\n");
}
int main() {
    char op[16];
    int a, b, c;
    while (scanf("%15s", op) == 1) {
        if (!strcmp(op, "init") && scanf("%d %d %d", &a, &b, &c) == 3) P.init(a, b, c);
        else if (!strcmp(op, "reset")) P.reset();
        else if (!strcmp(op, "ensure") && scanf("%d %d", &a, &b) == 2) printf("E %d\n", P.ensure(a, b, 64) ? 1 : 0);
        else if (!strcmp(op, "share") && scanf("%d %d %d", &a, &b, &c) == 3) P.share(a, b, c);
        else if (!strcmp(op, "uploaded")) P.uploaded();
        else if (!strcmp(op, "dump")) dump();
    }
    return 0;
}
"""


@pytest.fixture(scope="module")
def pool_exe(tmp_path_factory):
    d = tmp_path_factory.mktemp("pool")
    src = d / "drv.cpp"
    src.write_text(DRIVER)
    exe = d / "drv"
    subprocess.run(["g++", "-std=c++17", "-O1", "-I", CSRC, str(src), "-o", str(exe)], check=True)
    return str(exe)


def run(exe, script):
    out = subprocess.run([exe], input=script, capture_output=True, text=True, check=True).stdout.split("\n")
    ensures, dumps = [], []
    for line in out:
        if line.startswith("E "):
            ensures.append(int(line[2:]))
        elif line.startswith("T"):
            dumps.append({"table": [int(x) for x in line[1:].split()]})
        elif line.startswith("U "):
            u, cap, scr = (int(x) for x in line[2:].split())
            dumps[-1].update(in_use=u, capacity=cap, scratch=scr)
        elif line.startswith("D "):
            f = [int(x) for x in line[2:].split()]
            dumps[-1].update(full=f[0], pending=f[1:])
    return ensures, dumps


def test_pages_are_handed_out_in_order_and_never_twice(pool_exe):
    # 6 physical pages (5 usable + scratch 5), 3 slots of 4 entries
    ens, d = run(pool_exe, "init 6 3 4 dump uploaded ensure 0 70 ensure 1 10 ensure 0 100 ensure 0 129 dump")
    t0, t = d[0], d[1]
    assert t0["table"] == [5] * 12 and t0["full"] == 1 and t0["in_use"] == 0 and t0["capacity"] == 5
    assert ens == [1, 1, 1, 1]
    # slot 0: 70 tokens -> pages 0, 1; slot 1: page 2; slot 0 grows to 129 tokens -> page 3
    assert t["table"][:4] == [0, 1, 3, 5] and t["table"][4:8] == [2, 5, 5, 5] and t["table"][8:] == [5] * 4
    assert t["in_use"] == 4 and t["full"] == 0
    assert sorted(t["pending"]) == [0, 1, 2, 4]          # the entries assigned since the upload
    live = [p for p in t["table"] if p != t["scratch"]]
    assert len(live) == len(set(live))                    # no page backs two entries


def test_exhaustion_is_reported_and_reset_returns_everything(pool_exe):
    ens, d = run(pool_exe, "init 4 2 4 ensure 0 128 ensure 1 200 dump reset dump ensure 1 200 dump")
    assert ens[0] == 1 and ens[1] == 0                    # 3 usable pages: 2 + 4 do not fit
    t = d[0]
    assert t["in_use"] == 3 and t["table"][:2] == [0, 1] and t["table"][4] == 2 and t["table"][5] == 3
    assert d[1]["table"] == [3] * 8 and d[1]["in_use"] == 0 and d[1]["full"] == 1
    assert ens[2] == 0 and d[2]["table"][4:7] == [0, 1, 2]  # after the reset the same slot gets pages 0..2


def test_a_slot_never_takes_more_than_its_row(pool_exe):
    ens, d = run(pool_exe, "init 20 2 3 ensure 0 100000 dump")
    assert ens == [1] and d[0]["in_use"] == 3 and d[0]["table"][:3] == [0, 1, 2]


def test_shared_pages_for_the_training_blocks(pool_exe):
    # slot 0 holds 300 tokens (5 pages); slot 1's block starts at token 150: it shares slot 0's
    # first two pages and takes its own from logical page 2 on
    ens, d = run(pool_exe, "init 12 3 8 ensure 0 300 uploaded share 1 0 2 ensure 1 166 dump")
    t = d[0]
    assert ens == [1, 1]
    assert t["table"][8:11] == [0, 1, 5]                  # shared 0, 1; own page 5 for logical page 2
    assert sorted(t["pending"]) == [8, 9, 10]
    assert t["in_use"] == 6
