"""Model checks of the attention kernel's static unit schedules, on the CPU.

The kernel's roles (producer, MMA warps, softmax warps) all walk the same
sequence of units, given for CTA i of a grid of g by `unit_at` in
csrc/attn_fwd.cu; this module restates that function and the host's choice
between its two schedules, and checks over many shapes and grid sizes that

* every unit is processed exactly once (a unit left out would leave rows of
  O unwritten; one processed twice would only cost time, which no output
  comparison would show);
* the busiest CTA's key-tile count stays close to the mean: within one unit's
  length for the alternating rounds, within 1 % plus one item for the
  mirrored pairs where the host picks them;
* the mirrored-pair schedule keeps each round's items within two KV groups
  (the property that keeps K and V in L2)."""
import pytest


def host_paired(n_units, n_qt, causal, grid):
    items = n_units // 2
    rounds = (items + grid - 1) // grid
    return causal and n_qt % 2 == 0 and items >= 4 * grid and 100 * rounds * grid <= 101 * items


def unit_at(k, i, g, paired, B, Hkv, pairs, n_qt, n_units):
    if not paired:
        return k * g + ((g - 1 - i) if (k & 1) else i)
    half = n_qt // 2
    per_grp = half * pairs
    j = (k >> 1) * g + i
    if j >= B * Hkv * per_grp:
        return n_units
    grp, rem = divmod(j, per_grp)
    s, pr = divmod(rem, pairs)
    t = s if (k & 1) else n_qt - 1 - s
    return (n_qt - 1 - t) * (B * Hkv * pairs) + grp * pairs + pr


def decode(u, B, Hkv, pairs, n_qt):
    per_t = B * Hkv * pairs
    t = n_qt - 1 - u // per_t
    r = u % per_t
    b, r = divmod(r, Hkv * pairs)
    g, pr = divmod(r, pairs)
    return t, b, g, pr


def walk(B, Hkv, G, n_qt, grid, causal=True):
    pairs = (G + 1) // 2
    n_units = n_qt * B * Hkv * pairs
    g = min(n_units, grid)
    paired = host_paired(n_units, n_qt, causal, g)
    seen = [0] * n_units
    tiles = [0] * g
    rounds_groups = {}
    for i in range(g):
        k = 0
        while True:
            u = unit_at(k, i, g, paired, B, Hkv, pairs, n_qt, n_units)
            if u >= n_units:
                break
            seen[u] += 1
            t, b, kvg, _ = decode(u, B, Hkv, pairs, n_qt)
            tiles[i] += t + 1 if causal else n_qt
            rounds_groups.setdefault(k >> 1, set()).add(b * Hkv + kvg)
            k += 1
    return paired, seen, tiles, rounds_groups, n_qt + 1


SHAPES = [(B, Hkv, G, n_qt) for B in (1, 2, 3) for Hkv in (1, 2, 8) for G in (1, 2, 3, 4, 7)
          for n_qt in (1, 2, 7, 8, 64, 255, 256)]


@pytest.mark.parametrize("grid", [152, 148, 132, 7])
def test_every_unit_once(grid):
    for B, Hkv, G, n_qt in SHAPES:
        _, seen, _, _, _ = walk(B, Hkv, G, n_qt, grid)
        assert all(c == 1 for c in seen), (B, Hkv, G, n_qt, grid)


@pytest.mark.parametrize("grid", [152, 148, 132])
def test_balance(grid):
    for B, Hkv, G, n_qt in SHAPES:
        paired, _, tiles, _, item = walk(B, Hkv, G, n_qt, grid)
        if len(tiles) < grid:
            continue  # fewer units than CTAs: one unit each
        mean = sum(tiles) / len(tiles)
        if paired:
            assert max(tiles) <= 1.01 * mean + item, (B, Hkv, G, n_qt)
        else:
            assert max(tiles) <= mean + n_qt, (B, Hkv, G, n_qt)


def test_long_context_shape_takes_the_pairs_and_keeps_rounds_on_two_kv_groups():
    paired, seen, tiles, rounds_groups, _ = walk(2, 8, 4, 256, 152)
    assert paired
    assert all(len(gs) <= 2 for gs in rounds_groups.values())
    assert max(tiles) / (sum(tiles) / len(tiles)) < 1.003
