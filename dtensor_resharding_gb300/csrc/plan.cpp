// Host-side reshard planner: validation, shard boxes, replica groups, per-dim intersections,
// source choice and the device work-item tables.
//
// Follows the statement of the problem in the news article on NVIDIA's Reshard collective
// ("Recasting refit as a DTensor-to-DTensor transfer": the overlaps between source and
// destination shards are computable from the two DTensor descriptions; replication means one
// piece may be held by several sources) and the NeMo-RL design doc "NCCL Reshard Refit
// (Experimental)" ("xferdtensor Transports": compute the exact shard overlaps, move each
// destination region once, fan it out to the replicas; "Enabling It": one error listing every
// violation).
#include <algorithm>
#include <cstring>
#include <map>
#include <memory>
#include <new>
#include <sstream>
#include <utility>

#include "plan.h"

#ifndef RESHARD_SIZE_ORDER
#define RESHARD_SIZE_ORDER 1
#endif

namespace reshard {

namespace {
thread_local std::string g_error;
}

void set_error(const std::string &msg) { g_error = msg; }

int fail(int code, const std::string &msg) {
  g_error = msg;
  return code;
}

int64_t pointer_table_size(const reshard_plan *p) { return p->n_src_ptrs + 2 * p->n_dst_ptrs + 1; }

namespace {

int element_size(int dtype) {
  switch (dtype) {
    case RESHARD_U8: return 1;
    case RESHARD_BF16: return 2;
    case RESHARD_F16: return 2;
    case RESHARD_F32: return 4;
    case RESHARD_I32: return 4;
    case RESHARD_I64: return 8;
    default: return 0;
  }
}

// Validation messages collected across a whole batch; the strongest code wins.
struct Violations {
  std::vector<std::string> lines;
  int code = RESHARD_OK;
  void add(int c, const std::string &s) {
    lines.push_back(s);
    if (code == RESHARD_OK || c == RESHARD_ERR_INVALID_ARG) code = c;
  }
  int report() const {
    std::ostringstream o;
    o << lines.size() << " violation(s):";
    for (const auto &l : lines) o << "\n  " << l;
    return fail(code, o.str());
  }
};

int64_t volume(const Box &b, int nd) {
  int64_t v = 1;
  for (int d = 0; d < nd; ++d) v *= std::max<int64_t>(0, b.hi[d] - b.lo[d]);
  return v;
}

// The box owned by the rank at row-major mesh position `pos`: mesh dims are applied in
// order; Shard(d) on mesh dim k takes piece coord[k] of the current interval of dim d, split
// by torch.chunk's rule (pieces of ceil(len / n), trailing pieces possibly empty).
Box rank_box(const reshard_tensor_spec_t &s, const reshard_mesh_t &mesh, const reshard_placement_t *pl,
             int64_t pos) {
  Box b;
  for (int d = 0; d < kMaxDims; ++d) {
    b.lo[d] = 0;
    b.hi[d] = d < s.ndim ? s.global_shape[d] : 1;
  }
  int64_t coord[RESHARD_MAX_MESH_DIMS];
  for (int k = mesh.ndim - 1; k >= 0; --k) {
    coord[k] = pos % mesh.shape[k];
    pos /= mesh.shape[k];
  }
  for (int k = 0; k < mesh.ndim; ++k) {
    if (pl[k].kind != RESHARD_SHARD) continue;
    const int d = pl[k].dim;
    const int64_t len = b.hi[d] - b.lo[d];
    const int64_t n = mesh.shape[k];
    const int64_t piece = (len + n - 1) / n;  // torch.chunk piece length
    const int64_t start = std::min(len, coord[k] * piece);
    const int64_t stop = std::min(len, start + piece);
    b.hi[d] = b.lo[d] + stop;
    b.lo[d] = b.lo[d] + start;
  }
  return b;
}

void check_mesh(const char *side, const reshard_mesh_t &m, const reshard_placement_t *pl, int ndim,
                const std::string &pre, Violations &v) {
  if (m.ndim < 1 || m.ndim > RESHARD_MAX_MESH_DIMS) {
    v.add(RESHARD_ERR_UNSUPPORTED, pre + side + "_mesh.ndim must be in 1.." + std::to_string(RESHARD_MAX_MESH_DIMS));
    return;
  }
  if (!m.shape) {
    v.add(RESHARD_ERR_INVALID_ARG, pre + side + "_mesh.shape is NULL");
    return;
  }
  int64_t n = 1;
  for (int k = 0; k < m.ndim; ++k) {
    if (m.shape[k] < 1) v.add(RESHARD_ERR_INVALID_ARG, pre + side + "_mesh.shape[" + std::to_string(k) + "] < 1");
    n *= std::max<int64_t>(1, m.shape[k]);
  }
  if (n > (1 << 20)) v.add(RESHARD_ERR_UNSUPPORTED, pre + side + " mesh has more than 2^20 ranks");
  if (!pl) {
    v.add(RESHARD_ERR_INVALID_ARG, pre + side + " placements are NULL");
  } else {
    for (int k = 0; k < m.ndim; ++k) {
      if (pl[k].kind == RESHARD_REPLICATE) continue;
      if (pl[k].kind != RESHARD_SHARD)
        v.add(RESHARD_ERR_INVALID_ARG, pre + side + " placement " + std::to_string(k) + " has an unknown kind");
      else if (pl[k].dim < 0 || pl[k].dim >= ndim)
        v.add(RESHARD_ERR_INVALID_ARG, pre + side + " placement " + std::to_string(k) + " shards dim " +
                                           std::to_string(pl[k].dim) + " of a " + std::to_string(ndim) + "-d tensor");
    }
  }
  if (m.ranks && n <= (1 << 20)) {
    std::vector<char> seen((size_t)n, 0);
    for (int64_t i = 0; i < n; ++i) {
      const int32_t r = m.ranks[i];
      if (r < 0 || r >= n || seen[(size_t)r]) {
        v.add(RESHARD_ERR_INVALID_ARG, pre + side + "_mesh.ranks is not a permutation of 0.." + std::to_string(n - 1));
        break;
      }
      seen[(size_t)r] = 1;
    }
  }
}

// Fill boxes and views of one side (per pointer index) and check the views.
void side_layout(const reshard_tensor_spec_t &s, bool src, TensorInfo &t, const std::string &pre, Violations &v) {
  const reshard_mesh_t &m = src ? s.src_mesh : s.dst_mesh;
  const reshard_placement_t *pl = src ? s.src_pl : s.dst_pl;
  const reshard_view_t *views = src ? s.src_views : s.dst_views;
  const char *side = src ? "src" : "dst";
  int64_t n = 1;
  for (int k = 0; k < m.ndim; ++k) n *= m.shape[k];
  std::vector<Box> &boxes = src ? t.src_box : t.dst_box;
  std::vector<RankView> &rv = src ? t.src_view : t.dst_view;
  boxes.resize((size_t)n);
  rv.resize((size_t)n);
  for (int64_t pos = 0; pos < n; ++pos) {
    const int64_t p = m.ranks ? m.ranks[pos] : pos;
    boxes[(size_t)p] = rank_box(s, m, pl, pos);
  }
  for (int64_t p = 0; p < n; ++p) {
    const Box &b = boxes[(size_t)p];
    RankView &w = rv[(size_t)p];
    int64_t ext[kMaxDims];
    for (int d = 0; d < s.ndim; ++d) ext[d] = b.hi[d] - b.lo[d];
    int64_t dense = 1;
    for (int d = s.ndim - 1; d >= 0; --d) {
      w.strides[d] = dense;
      dense *= ext[d];
    }
    int64_t capacity = 0;
    if (views) {
      const reshard_view_t &vw = views[p];
      w.offset = vw.offset_elems;
      capacity = vw.capacity_elems;
      if (vw.offset_elems < 0) v.add(RESHARD_ERR_INVALID_ARG, pre + side + " view " + std::to_string(p) + " has a negative offset");
      if (vw.strides_elems) {
        w.dense = false;
        for (int d = 0; d < s.ndim; ++d) {
          w.strides[d] = vw.strides_elems[d];
          if (w.strides[d] < 0)
            v.add(RESHARD_ERR_INVALID_ARG, pre + side + " view " + std::to_string(p) + " has a negative stride");
        }
        // a stride equal to the dense one everywhere is still dense
        int64_t dd = 1;
        bool same = true;
        for (int d = s.ndim - 1; d >= 0; --d) {
          if (ext[d] > 1 && w.strides[d] != dd) same = false;
          dd *= ext[d];
        }
        if (same) {
          w.dense = true;
          dd = 1;
          for (int d = s.ndim - 1; d >= 0; --d) {
            w.strides[d] = dd;
            dd *= ext[d];
          }
        }
      }
    }
    const int64_t vol = volume(b, s.ndim);
    if (capacity > 0 && vol > 0) {
      int64_t last = w.offset;
      for (int d = 0; d < s.ndim; ++d) last += (ext[d] - 1) * w.strides[d];
      if (last + 1 > capacity)
        v.add(RESHARD_ERR_INVALID_ARG, pre + side + " view " + std::to_string(p) + " overflows its buffer (needs " +
                                           std::to_string(last + 1) + " elements, capacity " + std::to_string(capacity) + ")");
    }
  }
}

struct BoxKey {
  int64_t v[2 * kMaxDims];
  bool operator<(const BoxKey &o) const { return std::lexicographical_compare(v, v + 2 * kMaxDims, o.v, o.v + 2 * kMaxDims); }
};

BoxKey key_of(const Box &b) {
  BoxKey k;
  for (int d = 0; d < kMaxDims; ++d) {
    k.v[2 * d] = b.lo[d];
    k.v[2 * d + 1] = b.hi[d];
  }
  return k;
}

// Cut one strided region into 2-D work items (rows x run). `ext` are the region extents,
// `so`/`ss` and `dof`/`ds` the element offset and strides on the source and destination side.
void emit_items(int nd, const int64_t *ext, int64_t so, const int64_t *ss, int64_t dof, const int64_t *ds,
                int32_t src, int32_t group, int esize, int64_t item_bytes, std::vector<Item> &out) {
  for (int d = 0; d < nd; ++d)
    if (ext[d] <= 0) return;
  // innermost run, merged outward while both sides stay contiguous
  int64_t run = ext[nd - 1];
  int k = nd - 2;
  while (k >= 0 && (ext[k] == 1 || (ss[k] == run && ds[k] == run))) {
    run *= ext[k];
    --k;
  }
  // next non-trivial dim becomes the row dim; further dims merge while their pitch is uniform
  while (k >= 0 && ext[k] == 1) --k;
  int64_t rows = 1, sp = 0, dp = 0;
  if (k >= 0) {
    rows = ext[k];
    sp = ss[k];
    dp = ds[k];
    --k;
    while (k >= 0 && (ext[k] == 1 || (ss[k] == rows * sp && ds[k] == rows * dp))) {
      rows *= ext[k];
      --k;
    }
  }
  // remaining outer dims [0, k] are walked explicitly
  int64_t idx[kMaxDims + 1] = {0, 0, 0, 0, 0};
  const int64_t run_bytes = run * esize;
  for (;;) {
    int64_t s0 = so, d0 = dof;
    for (int d = 0; d <= k; ++d) {
      s0 += idx[d] * ss[d];
      d0 += idx[d] * ds[d];
    }
    Item it{};
    it.src = src;
    it.group = group;
    it.esize = esize;
    if (run_bytes > item_bytes) {
      int64_t seg = (item_bytes / esize) / kRunSplitElems * kRunSplitElems;
      if (seg < kRunSplitElems) seg = kRunSplitElems;
      for (int64_t r = 0; r < rows; ++r)
        for (int64_t c = 0; c < run; c += seg) {
          it.rows = 1;
          it.run = (int32_t)std::min(seg, run - c);
          it.src_off = s0 + r * sp + c;
          it.dst_off = d0 + r * dp + c;
          it.src_pitch = it.run;
          it.dst_pitch = it.run;
          out.push_back(it);
        }
    } else {
      const int64_t per = std::max<int64_t>(1, item_bytes / std::max<int64_t>(1, run_bytes));
      for (int64_t r = 0; r < rows; r += per) {
        it.rows = (int32_t)std::min(per, rows - r);
        it.run = (int32_t)run;
        it.src_off = s0 + r * sp;
        it.dst_off = d0 + r * dp;
        it.src_pitch = rows > 1 ? sp : run;
        it.dst_pitch = rows > 1 ? dp : run;
        out.push_back(it);
      }
    }
    int d = k;
    for (; d >= 0; --d) {
      if (++idx[d] < ext[d]) break;
      idx[d] = 0;
    }
    if (d < 0) break;
  }
}

// Side A (the reader) of a region, for the TMA slab of transposing items: the region origin
// sits at coordinates a_lo[d] of a slab of extents a_ext[d] whose element (0, ..., 0) is at
// element offset a_base of pointer a_ptr.
struct ReadSide {
  int32_t ptr;
  int64_t base;
  const int64_t *lo;
  const int64_t *ext;
};

// Emit the work of one region between side A (offset so, strides sa) and side B (offset dof,
// strides sb). When both sides are contiguous along the same dim (or neither has a contiguous
// dim), the region is a strided copy: that dim becomes the run. When A is contiguous along one
// dim and B along another, the region is a transpose and becomes transposing items.
void emit_region(int nd, const int64_t *ext, int64_t so, const int64_t *sa, const ReadSide &ra, int64_t dof,
                 const int64_t *sb, int32_t group, int esize, int64_t item_bytes, std::vector<Item> &out,
                 std::vector<TItem> &tout, std::map<SlabSpec, int32_t> &slab_ids, std::vector<SlabSpec> &slabs) {
  int ua = -1, ub = -1;
  for (int d = 0; d < nd; ++d) {
    if (ext[d] > 1 && sa[d] == 1) ua = d;
    if (ext[d] > 1 && sb[d] == 1) ub = d;
  }
  if (ua >= 0 && ub >= 0 && ua != ub) {
    const int R = ub, C = ua;
    const int64_t tc = kTileRowBytes / esize;
    const int64_t rows_per = (int64_t)kItemTiles * kTileRows, cols_per = kItemTiles * tc;
    int outer[kMaxDims], no = 0;
    for (int d = 0; d < nd; ++d)
      if (d != R && d != C && ext[d] > 1) outer[no++] = d;
    int64_t idx[kMaxDims] = {0, 0, 0, 0};
    for (;;) {
      int64_t sbase = so, dbase = dof, slab_base = ra.base;
      for (int d = 0; d < nd; ++d) {
        if (d == R || d == C) continue;
        const int64_t o = ext[d] > 1 ? idx[d] : 0;
        sbase += o * sa[d];
        dbase += o * sb[d];
        slab_base += (ra.lo[d] + o) * sa[d];
      }
      SlabSpec sl{ra.ptr, esize, slab_base, ra.ext[C], ra.ext[R], sa[R]};
      auto f = slab_ids.find(sl);
      int32_t sid;
      if (f == slab_ids.end()) {
        sid = (int32_t)slabs.size();
        slab_ids[sl] = sid;
        slabs.push_back(sl);
      } else {
        sid = f->second;
      }
      for (int64_t r0 = 0; r0 < ext[R]; r0 += rows_per)
        for (int64_t c0 = 0; c0 < ext[C]; c0 += cols_per) {
          TItem t{};
          t.src_off = sbase + r0 * sa[R] + c0;
          t.dst_off = dbase + c0 * sb[C] + r0;
          t.src_pitch = sa[R];
          t.dst_pitch = sb[C];
          t.rows = (int32_t)std::min(rows_per, ext[R] - r0);
          t.cols = (int32_t)std::min(cols_per, ext[C] - c0);
          t.src = ra.ptr;
          t.group = group;
          t.esize = esize;
          const int64_t x = ra.lo[C] + c0, y = ra.lo[R] + r0;
          const bool fits = x < INT32_MAX && y < INT32_MAX && sl.cols < ((int64_t)1 << 32) && sl.rows < ((int64_t)1 << 32);
          t.map = fits ? sid : -1;
          t.x = fits ? (int32_t)x : 0;
          t.y = fits ? (int32_t)y : 0;
          tout.push_back(t);
        }
      int k = no - 1;
      for (; k >= 0; --k) {
        const int d = outer[k];
        if (++idx[d] < ext[d]) break;
        idx[d] = 0;
      }
      if (k < 0) break;
    }
    return;
  }
  // strided copy: the shared contiguous dim (or a virtual unit dim) goes last as the run
  const int run_dim = (ua >= 0 && ua == ub) ? ua : -1;
  int64_t pe[kMaxDims + 1], pa[kMaxDims + 1], pb[kMaxDims + 1];
  int m = 0;
  for (int d = 0; d < nd; ++d) {
    if (d == run_dim) continue;
    pe[m] = ext[d];
    pa[m] = sa[d];
    pb[m] = sb[d];
    ++m;
  }
  if (run_dim >= 0) {
    pe[m] = ext[run_dim];
    pa[m] = 1;
    pb[m] = 1;
  } else {
    pe[m] = 1;
    pa[m] = 1;
    pb[m] = 1;
  }
  ++m;
  emit_items(m, pe, so, pa, dof, pb, ra.ptr, group, esize, item_bytes, out);
}

int build(const reshard_tensor_spec_t *specs, int n, reshard_plan_t **out) {
  if (!out) return fail(RESHARD_ERR_INVALID_ARG, "out is NULL");
  *out = nullptr;
  if (n < 0 || (n > 0 && !specs)) return fail(RESHARD_ERR_INVALID_ARG, "specs is NULL or n_tensors < 0");
  Violations v;
  std::unique_ptr<reshard_plan> owner(new reshard_plan());
  reshard_plan *plan = owner.get();
  plan->tensors.resize((size_t)n);

  // 1. validate every tensor and compute every rank's box and view
  for (int ti = 0; ti < n; ++ti) {
    const reshard_tensor_spec_t &s = specs[ti];
    const std::string pre = "tensor " + std::to_string(ti) + ": ";
    TensorInfo &t = plan->tensors[(size_t)ti];
    bool ok = true;
    if (s.ndim < 1 || s.ndim > kMaxDims) {
      v.add(RESHARD_ERR_UNSUPPORTED, pre + "ndim must be in 1.." + std::to_string(kMaxDims));
      ok = false;
    } else if (!s.global_shape) {
      v.add(RESHARD_ERR_INVALID_ARG, pre + "global_shape is NULL");
      ok = false;
    } else {
      for (int d = 0; d < s.ndim; ++d)
        if (s.global_shape[d] < 0) {
          v.add(RESHARD_ERR_INVALID_ARG, pre + "global_shape[" + std::to_string(d) + "] < 0");
          ok = false;
        }
    }
    t.esize = element_size(s.dtype);
    if (!t.esize) {
      v.add(RESHARD_ERR_INVALID_ARG, pre + "unknown dtype " + std::to_string(s.dtype));
      ok = false;
    }
    const size_t before = v.lines.size();
    check_mesh("src", s.src_mesh, s.src_pl, ok ? s.ndim : kMaxDims, pre, v);
    check_mesh("dst", s.dst_mesh, s.dst_pl, ok ? s.ndim : kMaxDims, pre, v);
    if (!ok || v.lines.size() != before) continue;
    t.ndim = s.ndim;
    t.dtype = s.dtype;
    for (int d = 0; d < s.ndim; ++d) t.shape[d] = s.global_shape[d];
    side_layout(s, true, t, pre, v);
    side_layout(s, false, t, pre, v);
    t.n_src = (int64_t)t.src_box.size();
    t.n_dst = (int64_t)t.dst_box.size();
    t.src_base = plan->n_src_ptrs;
    t.dst_base = plan->n_dst_ptrs;
    plan->n_src_ptrs += t.n_src;
    plan->n_dst_ptrs += t.n_dst;
  }
  if (!v.lines.empty()) return v.report();

  // 2. replica groups, intersections and source choice
  plan->quant_ok = true;
  auto quant_no = [&](const std::string &why) {
    if (plan->quant_ok) plan->quant_why = why;
    plan->quant_ok = false;
  };
  for (int ti = 0; ti < n; ++ti) {
    TensorInfo &t = plan->tensors[(size_t)ti];
    const int nd = t.ndim;
    const std::string pre = "tensor " + std::to_string(ti) + ": ";
    if (t.dtype != RESHARD_BF16) quant_no(pre + "MXFP8 needs a BF16 tensor");
    for (int64_t p = 0; p < t.n_src; ++p) {
      const Box &b = t.src_box[(size_t)p];
      if (volume(b, nd) > 0 && b.hi[nd - 1] - b.lo[nd - 1] > 1 && t.src_view[(size_t)p].strides[nd - 1] != 1)
        quant_no(pre + "MXFP8 needs sources contiguous along the last dim");
    }
    // source groups: identical boxes hold identical data; the lowest pointer index supplies
    std::map<BoxKey, int32_t> src_rep;
    for (int64_t p = 0; p < t.n_src; ++p) {
      if (volume(t.src_box[(size_t)p], nd) == 0) continue;
      auto k = key_of(t.src_box[(size_t)p]);
      if (!src_rep.count(k)) src_rep[k] = (int32_t)p;
    }
    std::vector<int32_t> reps;
    for (auto &kv : src_rep) reps.push_back(kv.second);
    std::sort(reps.begin(), reps.end());
    // destination groups: identical boxes and identical strides (offsets may differ)
    std::map<std::pair<BoxKey, std::vector<int64_t>>, int32_t> dst_gid;
    const int32_t first_group = (int32_t)plan->groups.size();
    for (int64_t p = 0; p < t.n_dst; ++p) {
      const Box &b = t.dst_box[(size_t)p];
      if (volume(b, nd) == 0) continue;
      const RankView &w = t.dst_view[(size_t)p];
      std::vector<int64_t> st(w.strides, w.strides + nd);
      auto key = std::make_pair(key_of(b), st);
      auto it = dst_gid.find(key);
      if (it == dst_gid.end()) {
        dst_gid[key] = (int32_t)plan->groups.size();
        Group g;
        g.tensor = ti;
        g.box = b;
        g.members.push_back((int32_t)p);
        plan->groups.push_back(g);
      } else {
        plan->groups[(size_t)it->second].members.push_back((int32_t)p);
      }
      if (!w.dense) quant_no(pre + "MXFP8 needs dense destination views");
      if (w.offset % 32) quant_no(pre + "MXFP8 destination offsets must be multiples of 32");
      if ((b.hi[nd - 1] - b.lo[nd - 1]) % 32) quant_no(pre + "MXFP8 needs every destination's last dim to be a multiple of 32");
    }
    for (int32_t g = first_group; g < (int32_t)plan->groups.size(); ++g) {
      Group &grp = plan->groups[(size_t)g];
      int64_t covered = 0;
      for (int32_t s : reps) {
        const Box &a = t.src_box[(size_t)s];
        Region r;
        r.tensor = ti;
        r.src = s;
        r.group = g;
        bool empty = false;
        for (int d = 0; d < kMaxDims; ++d) {
          r.box.lo[d] = std::max(a.lo[d], grp.box.lo[d]);
          r.box.hi[d] = std::min(a.hi[d], grp.box.hi[d]);
          if (d < nd && r.box.hi[d] <= r.box.lo[d]) empty = true;
        }
        if (empty) continue;
        covered += volume(r.box, nd);
        const int64_t c0 = r.box.lo[nd - 1] - grp.box.lo[nd - 1];
        const int64_t cw = r.box.hi[nd - 1] - r.box.lo[nd - 1];
        if (c0 % 32 || cw % 32) quant_no(pre + "MXFP8 blocks would straddle two sources (region edge not a multiple of 32)");
        plan->regions.push_back(r);
      }
      if (covered != volume(grp.box, nd)) {
        return fail(RESHARD_ERR_COVERAGE, pre + "sources cover " + std::to_string(covered) + " of " +
                                              std::to_string(volume(grp.box, nd)) + " destination elements");
      }
    }
  }
  if (n == 0) plan->quant_ok = true;

  // 3. packed-mode message layout: one message per (source rank, destination group members),
  //    regions in plan order inside a message, each starting on a 16-byte boundary
  std::map<std::pair<int32_t, std::vector<int32_t>>, std::vector<size_t>> messages;
  for (size_t i = 0; i < plan->regions.size(); ++i) {
    const Region &r = plan->regions[i];
    messages[std::make_pair(r.src, plan->groups[(size_t)r.group].members)].push_back(i);
  }
  int64_t msg_bytes = 0;
  for (auto &kv : messages)
    for (size_t i : kv.second) {
      Region &r = plan->regions[i];
      const TensorInfo &t = plan->tensors[(size_t)r.tensor];
      r.msg_off_bytes = msg_bytes;
      msg_bytes += (volume(r.box, t.ndim) * t.esize + 15) / 16 * 16;
    }

  // 4. group table (device layout) and the workspace pseudo-group
  const int64_t Ns = plan->n_src_ptrs, Nd = plan->n_dst_ptrs;
  plan->workspace_ptr = Ns + 2 * Nd;
  plan->grp_start.push_back(0);
  for (const Group &g : plan->groups) {
    const TensorInfo &t = plan->tensors[(size_t)g.tensor];
    for (int32_t m : g.members) {
      plan->mem_ptr.push_back((int32_t)(Ns + t.dst_base + m));
      plan->mem_off.push_back(t.dst_view[(size_t)m].offset);
    }
    plan->grp_start.push_back((int32_t)plan->mem_ptr.size());
    plan->max_fanout = std::max(plan->max_fanout, (int)g.members.size());
  }
  plan->workspace_group = (int32_t)plan->groups.size();
  plan->mem_ptr.push_back((int32_t)plan->workspace_ptr);
  plan->mem_off.push_back(0);
  plan->grp_start.push_back((int32_t)plan->mem_ptr.size());

  // 5. work items: direct (source -> destination replicas), pack (source -> message),
  //    unpack (message -> destination replicas)
  int64_t bytes_read = 0, bytes_written = 0, global_bytes = 0;
  int64_t plan_bytes = 0;
  for (const Region &r : plan->regions)
    plan_bytes += volume(r.box, plan->tensors[(size_t)r.tensor].ndim) * plan->tensors[(size_t)r.tensor].esize;
  int64_t item_bytes = kMaxItemBytes;
  while (item_bytes > kMinItemBytes && plan_bytes / item_bytes < kItemsPerPlan) item_bytes /= 2;
  std::map<SlabSpec, int32_t> slab_ids;
  for (const Region &r : plan->regions) {
    const TensorInfo &t = plan->tensors[(size_t)r.tensor];
    const int nd = t.ndim;
    const Box &sb = t.src_box[(size_t)r.src];
    const Group &g = plan->groups[(size_t)r.group];
    const RankView &sv = t.src_view[(size_t)r.src];
    const RankView &dv = t.dst_view[(size_t)g.members[0]];
    int64_t ext[kMaxDims], ms[kMaxDims];
    int64_t so = sv.offset, dof = 0;
    for (int d = 0; d < nd; ++d) {
      ext[d] = r.box.hi[d] - r.box.lo[d];
      so += (r.box.lo[d] - sb.lo[d]) * sv.strides[d];
      dof += (r.box.lo[d] - g.box.lo[d]) * dv.strides[d];
    }
    int64_t dd = 1;
    for (int d = nd - 1; d >= 0; --d) {
      ms[d] = dd;
      dd *= ext[d];
    }
    const int32_t sp = (int32_t)(t.src_base + r.src);
    const int64_t mo = r.msg_off_bytes / t.esize;
    int64_t slo[kMaxDims], sext[kMaxDims], zero[kMaxDims] = {0, 0, 0, 0};
    for (int d = 0; d < nd; ++d) {
      slo[d] = r.box.lo[d] - sb.lo[d];
      sext[d] = sb.hi[d] - sb.lo[d];
    }
    const ReadSide from_src{sp, sv.offset, slo, sext};
    const ReadSide from_msg{(int32_t)plan->workspace_ptr, mo, zero, ext};
    emit_region(nd, ext, so, sv.strides, from_src, dof, dv.strides, r.group, t.esize, item_bytes,
                plan->items[kDirect], plan->titems[kDirect], slab_ids, plan->slabs);
    emit_region(nd, ext, so, sv.strides, from_src, mo, ms, plan->workspace_group, t.esize, item_bytes,
                plan->items[kPack], plan->titems[kPack], slab_ids, plan->slabs);
    emit_region(nd, ext, mo, ms, from_msg, dof, dv.strides, r.group, t.esize, item_bytes, plan->items[kUnpack],
                plan->titems[kUnpack], slab_ids, plan->slabs);
    const int64_t b = volume(r.box, nd) * t.esize;
    bytes_read += b;
    bytes_written += b * (int64_t)g.members.size();
  }
#if RESHARD_SIZE_ORDER
  // largest items first: the persistent grid deals items round-robin, so CTAs finish together
  for (auto &iv : plan->items)
    std::stable_sort(iv.begin(), iv.end(), [](const Item &a, const Item &b) {
      return (int64_t)a.rows * a.run * a.esize > (int64_t)b.rows * b.run * b.esize;
    });
#endif
  // transposing items grouped by element size: the executor launches one build of its
  // transposing kernel per element size present, each over a contiguous run of the table
  for (auto &tv : plan->titems)
    std::stable_sort(tv.begin(), tv.end(), [](const TItem &a, const TItem &b) { return a.esize < b.esize; });
  for (const TensorInfo &t : plan->tensors) {
    int64_t v2 = t.esize;
    for (int d = 0; d < t.ndim; ++d) v2 *= t.shape[d];
    global_bytes += v2;
  }

  reshard_stats_t &st = plan->stats;
  st.n_tensors = n;
  st.regions = (int64_t)plan->regions.size();
  st.items = (int64_t)(plan->items[kDirect].size() + plan->titems[kDirect].size());
  st.dst_groups = (int64_t)plan->groups.size();
  st.messages = (int64_t)messages.size();
  st.bytes_read = bytes_read;
  st.bytes_written = bytes_written;
  st.wire_bytes = bytes_read;
  st.message_bytes = msg_bytes;
  st.gather_bcast_bytes = 2 * global_bytes;
  st.global_bytes = global_bytes;
  if (st.items > INT32_MAX || (int64_t)plan->mem_ptr.size() > INT32_MAX || (int64_t)plan->slabs.size() > INT32_MAX ||
      pointer_table_size(plan) > INT32_MAX) {
    return fail(RESHARD_ERR_UNSUPPORTED, "plan too large (more than 2^31 items, members or pointers)");
  }
  *out = owner.release();
  set_error("");
  return RESHARD_OK;
}

}  // namespace
}  // namespace reshard

using namespace reshard;

extern "C" int reshard_plan_create(const reshard_tensor_spec_t *spec, reshard_plan_t **out) {
  if (!spec) return fail(RESHARD_ERR_INVALID_ARG, "spec is NULL");
  try {
    return build(spec, 1, out);
  } catch (const std::bad_alloc &) {
    return fail(RESHARD_ERR_OOM, "host allocation failed while planning");
  }
}

extern "C" int reshard_plan_batch(const reshard_tensor_spec_t *specs, int n_tensors, reshard_plan_t **out) {
  try {
    return build(specs, n_tensors, out);
  } catch (const std::bad_alloc &) {
    return fail(RESHARD_ERR_OOM, "host allocation failed while planning");
  }
}

extern "C" int reshard_plan_blockwise_fp8(const reshard_tensor_spec_t *specs, int n, int64_t block_rows,
                                          int64_t block_cols, reshard_plan_t **out) {
  if (!out) return fail(RESHARD_ERR_INVALID_ARG, "out is NULL");
  *out = nullptr;
  if (n < 0 || (n > 0 && !specs)) return fail(RESHARD_ERR_INVALID_ARG, "specs is NULL or n_tensors < 0");
  if (block_rows < 1 || block_cols < 1) return fail(RESHARD_ERR_INVALID_ARG, "block sizes must be >= 1");
  try {
    Violations v;
    std::vector<reshard_tensor_spec_t> all(specs, specs + n);
    std::vector<std::vector<int64_t>> shapes((size_t)n);
    for (int i = 0; i < n; ++i) {
      const reshard_tensor_spec_t &d = specs[i];
      const std::string pre = "tensor " + std::to_string(i) + ": ";
      if (d.dtype != RESHARD_U8) v.add(RESHARD_ERR_INVALID_ARG, pre + "blockwise FP8 weights are RESHARD_U8");
      if (d.ndim < 2 || d.ndim > kMaxDims || !d.global_shape) {
        v.add(RESHARD_ERR_INVALID_ARG, pre + "blockwise FP8 weights need 2..4 dims");
        continue;
      }
      shapes[(size_t)i].assign(d.global_shape, d.global_shape + d.ndim);
      auto &sh = shapes[(size_t)i];
      sh[(size_t)d.ndim - 2] = (sh[(size_t)d.ndim - 2] + block_rows - 1) / block_rows;
      sh[(size_t)d.ndim - 1] = (sh[(size_t)d.ndim - 1] + block_cols - 1) / block_cols;
    }
    if (!v.lines.empty()) return v.report();
    for (int i = 0; i < n; ++i) {
      reshard_tensor_spec_t sc = specs[i];
      sc.global_shape = shapes[(size_t)i].data();
      sc.dtype = RESHARD_F32;
      sc.src_views = nullptr;
      sc.dst_views = nullptr;
      all.push_back(sc);
    }
    // every weight shard boundary on a block boundary, and every scale shard = its blocks
    for (int i = 0; i < n; ++i) {
      const reshard_tensor_spec_t &d = specs[i];
      const reshard_tensor_spec_t &sc = all[(size_t)(n + i)];
      for (int side = 0; side < 2; ++side) {
        const reshard_mesh_t &m = side ? d.dst_mesh : d.src_mesh;
        const reshard_placement_t *pl = side ? d.dst_pl : d.src_pl;
        if (m.ndim < 1 || m.ndim > RESHARD_MAX_MESH_DIMS || !m.shape || !pl) continue;  // reported by build
        int64_t nr = 1;
        for (int k = 0; k < m.ndim; ++k) nr *= std::max<int64_t>(1, m.shape[k]);
        for (int64_t pos = 0; pos < nr; ++pos) {
          const Box db = rank_box(d, m, pl, pos), sb = rank_box(sc, m, pl, pos);
          for (int k = 0; k < 2; ++k) {
            const int dim = d.ndim - 2 + k;
            const int64_t bs = k ? block_cols : block_rows, L = d.global_shape[dim];
            const bool lo_ok = db.lo[dim] % bs == 0 && sb.lo[dim] == db.lo[dim] / bs;
            const bool hi_ok = (db.hi[dim] % bs == 0 || db.hi[dim] == L) && sb.hi[dim] == (db.hi[dim] + bs - 1) / bs;
            const bool empty = db.hi[dim] == db.lo[dim] && sb.hi[dim] == sb.lo[dim];
            if (!empty && !(lo_ok && hi_ok)) {
              v.add(RESHARD_ERR_UNSUPPORTED, "tensor " + std::to_string(i) + ": " + (side ? "destination" : "source") +
                                                 " rank " + std::to_string(pos) + " splits dim " + std::to_string(dim) +
                                                 " off the " + std::to_string(bs) + "-element block grid");
              pos = nr;  // one line per tensor side
              break;
            }
          }
        }
      }
    }
    if (!v.lines.empty()) return v.report();
    return build(all.data(), (int)all.size(), out);
  } catch (const std::bad_alloc &) {
    return fail(RESHARD_ERR_OOM, "host allocation failed while planning");
  }
}

extern "C" int reshard_plan_stats(const reshard_plan_t *plan, reshard_stats_t *out) {
  if (!plan || !out) return fail(RESHARD_ERR_INVALID_ARG, "plan or out is NULL");
  *out = plan->stats;
  out->last_launches = plan->last_launches;
  out->last_aligned_items = plan->last_aligned;
  out->last_general_items = plan->last_general;
  out->last_rows_kernel = plan->last_rows_kernel;
  return RESHARD_OK;
}

extern "C" int reshard_plan_regions(const reshard_plan_t *plan, int64_t cap, int32_t *tensor, int32_t *src_rank,
                                    int32_t *dst_group, int64_t *lo, int64_t *hi, int64_t *n_out) {
  if (!plan) return fail(RESHARD_ERR_INVALID_ARG, "plan is NULL");
  const int64_t n = (int64_t)plan->regions.size();
  if (n_out) *n_out = n;
  for (int64_t i = 0; i < std::min(n, cap); ++i) {
    const Region &r = plan->regions[(size_t)i];
    if (tensor) tensor[i] = r.tensor;
    if (src_rank) src_rank[i] = r.src;
    if (dst_group) dst_group[i] = r.group;
    for (int d = 0; d < kMaxDims; ++d) {
      if (lo) lo[i * kMaxDims + d] = r.box.lo[d];
      if (hi) hi[i * kMaxDims + d] = r.box.hi[d];
    }
  }
  return RESHARD_OK;
}

extern "C" int reshard_plan_group_members(const reshard_plan_t *plan, int64_t g, int64_t cap, int32_t *members,
                                          int64_t *n_out) {
  if (!plan) return fail(RESHARD_ERR_INVALID_ARG, "plan is NULL");
  if (g < 0 || g >= (int64_t)plan->groups.size()) return fail(RESHARD_ERR_INVALID_ARG, "group out of range");
  const auto &m = plan->groups[(size_t)g].members;
  if (n_out) *n_out = (int64_t)m.size();
  for (int64_t i = 0; i < std::min<int64_t>(cap, (int64_t)m.size()); ++i)
    if (members) members[i] = m[(size_t)i];
  return RESHARD_OK;
}

extern "C" int reshard_plan_items(const reshard_plan_t *plan, int set, int64_t cap, void *items, int64_t *n_out,
                                  int32_t *group_start, int32_t *member_ptr, int64_t *member_off,
                                  int64_t *n_groups_out, int64_t *n_members_out) {
  if (!plan) return fail(RESHARD_ERR_INVALID_ARG, "plan is NULL");
  if (set < 0 || set >= 2 * kNumSets) return fail(RESHARD_ERR_INVALID_ARG, "set must be in 0..5");
  static_assert(sizeof(Item) == sizeof(TItem), "both item kinds are 64 bytes");
  const size_t count = set < kNumSets ? plan->items[set].size() : plan->titems[set - kNumSets].size();
  const void *data = set < kNumSets ? (const void *)plan->items[set].data() : (const void *)plan->titems[set - kNumSets].data();
  if (n_out) *n_out = (int64_t)count;
  if (items && cap > 0) std::memcpy(items, data, (size_t)std::min<int64_t>(cap, (int64_t)count) * sizeof(Item));
  if (n_groups_out) *n_groups_out = (int64_t)plan->grp_start.size() - 1;
  if (n_members_out) *n_members_out = (int64_t)plan->mem_ptr.size();
  if (group_start) std::memcpy(group_start, plan->grp_start.data(), plan->grp_start.size() * sizeof(int32_t));
  if (member_ptr) std::memcpy(member_ptr, plan->mem_ptr.data(), plan->mem_ptr.size() * sizeof(int32_t));
  if (member_off) std::memcpy(member_off, plan->mem_off.data(), plan->mem_off.size() * sizeof(int64_t));
  return RESHARD_OK;
}

extern "C" int reshard_plan_slabs(const reshard_plan_t *plan, int64_t cap, int64_t *out, int64_t *n_out) {
  if (!plan) return fail(RESHARD_ERR_INVALID_ARG, "plan is NULL");
  if (n_out) *n_out = (int64_t)plan->slabs.size();
  for (int64_t i = 0; i < std::min<int64_t>(cap, (int64_t)plan->slabs.size()); ++i) {
    const SlabSpec &s = plan->slabs[(size_t)i];
    int64_t *o = out + 6 * i;
    o[0] = s.ptr;
    o[1] = s.esize;
    o[2] = s.base_off;
    o[3] = s.cols;
    o[4] = s.rows;
    o[5] = s.pitch;
  }
  return RESHARD_OK;
}

extern "C" const char *reshard_last_error(void) { return g_error.c_str(); }
