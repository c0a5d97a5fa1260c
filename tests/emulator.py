"""Host emulation of the device work-item tables, for CPU tests (plain copies, no quantization).

Each copy item moves `rows` rows of `run` elements from its source pointer to every member of
its group; each transposing item moves element (r, c) from src_off + r * src_pitch + c to
member offset + dst_off + c * dst_pitch + r; each gather item writes `rows` destination rows of
run[0] + run[1] elements, piece 0's elements then piece 1's, each piece read from its own source
pointer. Pointer-table entries are given as (array name, byte offset of the entry's buffer in
that array, end offset).
"""
import numpy as np

import dtensor_resharding_gb300 as R


def run_items(plan, which, table, arrays, gather=False):
    """Apply pass `which` (0 direct, 1 pack, 2 unpack) of `plan` to the named host arrays. With
    `gather`, the pass runs as the executor runs it when it has gather items: the gather items,
    and the copy items they do not cover (pad[0] == 0)."""
    items, gs, mp, mo = R.reshard_plan_items(plan, which + 3)
    for it in items:
        e = int(it["esize"])
        kind, base, _ = table[it["src"]]
        rr, cc = np.meshgrid(np.arange(int(it["rows"])), np.arange(int(it["cols"])), indexing="ij")
        soff = base + (int(it["src_off"]) + rr * int(it["src_pitch"]) + cc) * e
        vals = arrays[kind][(soff[..., None] + np.arange(e)).reshape(-1)]
        for m in range(gs[it["group"]], gs[it["group"] + 1]):
            dkind, dbase, _ = table[mp[m]]
            doff = dbase + (int(mo[m]) + int(it["dst_off"]) + cc * int(it["dst_pitch"]) + rr) * e
            arrays[dkind][(doff[..., None] + np.arange(e)).reshape(-1)] = vals
    skip_flagged = False
    if gather:
        gitems, gs, mp, mo = R.reshard_plan_items(plan, 6 + which)
        skip_flagged = len(gitems) > 0
        for it in gitems:
            e = int(it["esize"])
            n0, n1 = int(it["run"][0]) * e, int(it["run"][1]) * e
            k0, b0, _ = table[it["src"][0]]
            k1, b1, _ = table[it["src"][1]]
            for m in range(gs[it["group"]], gs[it["group"] + 1]):
                dkind, dbase, _ = table[mp[m]]
                darr = arrays[dkind]
                for r in range(int(it["rows"])):
                    s0 = b0 + (int(it["src_off"][0]) + r * int(it["src_pitch"][0])) * e
                    s1 = b1 + (int(it["src_off"][1]) + r * int(it["src_pitch"][1])) * e
                    d0 = dbase + (int(mo[m]) + int(it["dst_off"]) + r * int(it["dst_pitch"])) * e
                    darr[d0: d0 + n0] = arrays[k0][s0: s0 + n0]
                    darr[d0 + n0: d0 + n0 + n1] = arrays[k1][s1: s1 + n1]
    items, gs, mp, mo = R.reshard_plan_items(plan, which)
    for it in items:
        if skip_flagged and int(it["pad"][0]) == 1:
            continue
        e = int(it["esize"])
        kind, base, _ = table[it["src"]]
        sarr = arrays[kind]
        for m in range(gs[it["group"]], gs[it["group"] + 1]):
            dkind, dbase, _ = table[mp[m]]
            darr = arrays[dkind]
            for r in range(int(it["rows"])):
                s0 = base + (int(it["src_off"]) + r * int(it["src_pitch"])) * e
                d0 = dbase + (int(mo[m]) + int(it["dst_off"]) + r * int(it["dst_pitch"])) * e
                n = int(it["run"]) * e
                darr[d0: d0 + n] = sarr[s0: s0 + n]
