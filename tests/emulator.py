"""Host emulation of the device work-item tables, for CPU tests (plain copies, no quantization).

Each copy item moves `rows` rows of `run` elements from its source pointer to every member of
its group; each transposing item moves element (r, c) from src_off + r * src_pitch + c to
member offset + dst_off + c * dst_pitch + r; each pair item moves `rows` rows of its two pieces,
piece p's run[p] elements from src_off[p] + r * src_pitch[p] of pointer src[p] to member offset +
dst_off[p] + r * dst_pitch[p] of every member (a gather row's pieces land side by side in one
destination row, a scatter row's in two message blocks). Pointer-table entries are given as
(array name, byte offset of the entry's buffer in that array, end offset).
"""
import numpy as np

import dtensor_resharding_gb300 as R


def run_items(plan, which, table, arrays, gather=False):
    """Apply pass `which` (0 direct, 1 pack, 2 unpack) of `plan` to the named host arrays. With
    `gather`, the pass runs as the executor runs it when it has pair items: the pair items, and
    the copy items they do not cover (pad[0] == 0)."""
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
            for m in range(gs[it["group"]], gs[it["group"] + 1]):
                dkind, dbase, _ = table[mp[m]]
                darr = arrays[dkind]
                for q in (0, 1):
                    n = int(it["run"][q]) * e
                    sk, sb, _ = table[it["src"][q]]
                    for r in range(int(it["rows"])):
                        s0 = sb + (int(it["src_off"][q]) + r * int(it["src_pitch"][q])) * e
                        d0 = dbase + (int(mo[m]) + int(it["dst_off"][q]) + r * int(it["dst_pitch"][q])) * e
                        darr[d0: d0 + n] = arrays[sk][s0: s0 + n]
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
