"""Host-side invariants of the skinny kernel's stream-K partition (no GPU).

In stream-K mode the kernel gives CTA c the units [c U / G, (c+1) U / G) of
the U = n_cb * n_kb (column group, 64-deep k-block) units, G CTAs in all.
Each CTA writes one partial sum per column group it touches, into slot
(c - c_lo) of that group, c_lo being the group's first CTA.  The plan must
therefore give every group at least as many slots as the most CTAs whose
ranges meet one group's k-blocks, and the workspace must hold all the slots
and the groups' arrival counters.  These tests rebuild the partition from
its definition and check the library's plans against it.
"""
import random

import pytest

import swiglu_mlp_projection_gb300 as swg


def cta_of(t, U, G):
    # the CTA whose range [c U / G, (c+1) U / G) holds unit t
    return ((t + 1) * G + U - 1) // U - 1


def max_contributors(U, G, n_kb, n_cb):
    worst = 0
    for g in range(n_cb):
        lo, hi = cta_of(g * n_kb, U, G), cta_of((g + 1) * n_kb - 1, U, G)
        worst = max(worst, hi - lo + 1)
    return worst


def geometry(M, K, n_out, nb, plain, num_sms):
    n = 16
    while n < M:
        n *= 2
    while nb > 1 and nb * n > 256:
        nb //= 2
    sub_cols = 128 if plain else 64
    n_cb = -(-(-(-n_out // sub_cols)) // nb)
    n_kb = -(-K // 64)
    units = n_cb * n_kb
    return nb, n_cb, n_kb, units, max(1, min(units, num_sms))


def test_cta_of_matches_the_ranges():
    for U, G in [(1, 1), (7, 3), (100, 7), (3584, 152), (152, 152), (151, 152)]:
        G = min(G, U)
        for c in range(G):
            for t in range(c * U // G, (c + 1) * U // G):
                assert cta_of(t, U, G) == c


@pytest.mark.parametrize("nb", [1, 2, 4])
@pytest.mark.parametrize("op", ["up", "down"])
def test_slots_cover_every_group(cuda_lib, monkeypatch, nb, op):
    monkeypatch.setenv("SWIGLU_SK_CLUSTER", "0")   # stream-K mode
    monkeypatch.setenv("SWIGLU_SK_NB", str(nb))
    rng = random.Random(nb * 10 + (op == "down"))
    shapes = [(1, 4096, 14336), (16, 4096, 14336), (64, 4096, 14336), (128, 8192, 29568),
              (256, 896, 4864), (3, 64, 8), (17, 520, 1032)]
    shapes += [(rng.randint(1, 256), 8 * rng.randint(1, 2048), 8 * rng.randint(1, 4096))
               for _ in range(60)]
    for M, d, d_ff in shapes:
        for num_sms in (152, 132, 20):
            if op == "up":
                p = swg.plan(M, d, d_ff, "bf16", "skinny", num_sms)
                K, n_out, plain = d, d_ff, False
            else:
                p = swg.down_plan(M, d_ff, d, "bf16", "skinny", num_sms)
                K, n_out, plain = d_ff, d, True
            nb_eff, n_cb, n_kb, units, grid = geometry(M, K, n_out, nb, plain, num_sms)
            assert p["path"] == "skinny" and p["cluster"] == 1
            assert p["grid"] == grid, (M, d, d_ff, num_sms)
            need = max_contributors(units, grid, n_kb, n_cb)
            assert p["slices"] >= need, (M, d, d_ff, num_sms, p["slices"], need)
            partials = n_cb * p["slices"] * nb_eff * 2 * M * 64 * 4
            assert p["workspace"] >= partials + 4 * n_cb, (M, d, d_ff, num_sms)


def slots(units, grid, n_kb):
    # the plan's slot count: a group's k-blocks meet at most this many CTAs
    per = units // grid
    return -(-n_kb // per) + 1


@pytest.mark.parametrize("split", ["default", "0"])
def test_down_projection_column_group_rule(cuda_lib, split, monkeypatch):
    # No override, sums in a second kernel (the bf16 default): 256-column
    # groups up to 128 rows (64 above 256 MB of weights), 128-column groups
    # above.  With the group's last
    # CTA adding the sums (SWIGLU_SK_SPLIT=0): 128-column groups once
    # 256-column groups would collect more than 256 KB of partial sums per
    # group (slots x 256 columns x M x 4 B).  Either way every group has
    # enough slots.
    if split == "0":
        monkeypatch.setenv("SWIGLU_SK_SPLIT", "0")
    for M in (1, 8, 16, 24, 32, 48, 49, 64, 96, 128, 256):
        for d, d_ff in ((4096, 14336), (8192, 29568)):
            p = swg.down_plan(M, d_ff, d, "bf16", "skinny", 152)
            assert p["cluster"] == 1 and p["launches"] == (1 if split == "0" else 2)
            _, _, n_kb2, units2, grid2 = geometry(M, d_ff, d, 2, True, 152)
            if split == "0":
                nb = 1 if slots(units2, grid2, n_kb2) * 256 * 4 * M > 256 * 1024 else 2
            else:
                nb = 1 if M > (64 if d_ff * d * 2 > 256 << 20 else 128) else 2
            _, n_cb, n_kb, units, grid = geometry(M, d_ff, d, nb, True, 152)
            assert p["slices"] == slots(units, grid, n_kb), (M, d, nb)
            assert p["slices"] >= max_contributors(units, grid, n_kb, n_cb)
