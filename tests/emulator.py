"""Host emulation of the device work-item tables, for CPU tests (plain copies, no quantization).

Each copy item moves `rows` rows of `run` elements from its source pointer to every member of
its group; each transposing item moves element (r, c) from src_off + r * src_pitch + c to
member offset + dst_off + c * dst_pitch + r. Pointer-table entries are given as
(array name, byte offset of the entry's buffer in that array, end offset).
"""
import numpy as np

import dtensor_resharding_gb300 as R


def run_items(plan, which, table, arrays):
    """Apply pass `which` (0 direct, 1 pack, 2 unpack) of `plan` to the named host arrays."""
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
    items, gs, mp, mo = R.reshard_plan_items(plan, which)
    for it in items:
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
