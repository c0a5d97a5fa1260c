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

int64_t pointer_table_size(const reshard_plan *p) { return p->n_src_ptrs + 2 * p->n_dst_ptrs + 2; }

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
    // a destination's elements must have distinct offsets (else what it receives depends on
    // the order of the writes): taken by increasing stride, every dim's stride must pass the
    // span of the dims below it (views interleaving two dims otherwise are refused too)
    if (!src && !w.dense && vol > 1) {
      int order[kMaxDims], k = 0;
      for (int d = 0; d < s.ndim; ++d)
        if (ext[d] > 1) order[k++] = d;
      std::sort(order, order + k, [&](int x, int y) { return w.strides[x] < w.strides[y]; });
      int64_t span = 0;
      for (int q = 0; q < k; ++q) {
        const int d = order[q];
        if (w.strides[d] <= span) {
          v.add(RESHARD_ERR_INVALID_ARG, pre + side + " view " + std::to_string(p) + " maps two elements to one offset (stride " +
                                             std::to_string(w.strides[d]) + " of dim " + std::to_string(d) +
                                             " within the span of the smaller strides)");
          break;
        }
        span += w.strides[d] * (ext[d] - 1);
      }
    }
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

// Steps 1 and 2: validation, every rank's box and view, replica groups, intersections and the
// source of every region. Fills plan->tensors, regions, groups and the MXFP8 eligibility.
int plan_regions(const reshard_tensor_spec_t *specs, int n, reshard_plan *plan) {
  if (n < 0 || (n > 0 && !specs)) return fail(RESHARD_ERR_INVALID_ARG, "specs is NULL or n_tensors < 0");
  Violations v;
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
    t.src_rep.assign((size_t)t.n_src, -1);
    for (int64_t p = 0; p < t.n_src; ++p) {
      if (volume(t.src_box[(size_t)p], nd) == 0) continue;
      auto k = key_of(t.src_box[(size_t)p]);
      if (!src_rep.count(k)) src_rep[k] = (int32_t)p;
      t.src_rep[(size_t)p] = src_rep[k];
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
  return RESHARD_OK;
}

int64_t region_bytes(const reshard_plan &p, const Region &r) {
  const TensorInfo &t = p.tensors[(size_t)r.tensor];
  return volume(r.box, t.ndim) * t.esize;
}

int64_t align16(int64_t x) { return (x + 15) / 16 * 16; }

// Element offset of region r's origin in its source's buffer, and that source's view.
const RankView &region_source(const reshard_plan &p, const Region &r, int64_t &so) {
  const TensorInfo &t = p.tensors[(size_t)r.tensor];
  const Box &sb = t.src_box[(size_t)r.src];
  const RankView &sv = t.src_view[(size_t)r.src];
  so = sv.offset;
  for (int d = 0; d < t.ndim; ++d) so += (r.box.lo[d] - sb.lo[d]) * sv.strides[d];
  return sv;
}

// Element offset of region r's origin relative to a member of device group g (the members share
// strides; each adds its own view offset), and those strides.
const int64_t *region_dest(const reshard_plan &p, const Region &r, const Group &g, int64_t &dof) {
  const TensorInfo &t = p.tensors[(size_t)r.tensor];
  const RankView &dv = t.dst_view[(size_t)g.members[0]];
  dof = 0;
  for (int d = 0; d < t.ndim; ++d) dof += (r.box.lo[d] - g.box.lo[d]) * dv.strides[d];
  return dv.strides;
}

// Pack-pass pairs: regions read from the same source shard with the same box but for the last
// dim, region A ending where region B starts, both packed into messages (the send buffer), the
// last dim contiguous in the source, at least two elements of each piece and two rows: one
// source row feeds two message blocks. Only rows misaligned by construction pair up (a piece's
// bytes per row not a multiple of 16: its dense message rows are then misaligned). Same encoding
// of partner[] as gather_pairs.
std::vector<int64_t> scatter_pairs(const reshard_plan &p, const std::vector<Role> &roles) {
  std::vector<int64_t> partner(p.regions.size(), -1);
  std::map<std::vector<int64_t>, std::vector<size_t>> rows_of;
  for (size_t i = 0; i < p.regions.size(); ++i) {
    const Region &r = p.regions[i];
    const TensorInfo &t = p.tensors[(size_t)r.tensor];
    const int nd = t.ndim, last = nd - 1;
    if (roles[i].send_off < 0 || nd < 2) continue;
    if (r.box.hi[last] - r.box.lo[last] < 2 || r.box.hi[last - 1] - r.box.lo[last - 1] < 2) continue;
    if (t.src_view[(size_t)r.src].strides[last] != 1) continue;
    std::vector<int64_t> key{r.tensor, r.src};
    for (int d = 0; d < last; ++d) {
      key.push_back(r.box.lo[d]);
      key.push_back(r.box.hi[d]);
    }
    rows_of[key].push_back(i);
  }
  for (auto &kv : rows_of) {
    std::vector<size_t> &v = kv.second;
    if (v.size() < 2) continue;
    const TensorInfo &t = p.tensors[(size_t)p.regions[v[0]].tensor];
    const int last = t.ndim - 1;
    std::sort(v.begin(), v.end(), [&](size_t a, size_t b) { return p.regions[a].box.lo[last] < p.regions[b].box.lo[last]; });
    for (size_t k = 0; k + 1 < v.size(); ++k) {
      const Region &a = p.regions[v[k]], &b = p.regions[v[k + 1]];
      if (a.box.hi[last] != b.box.lo[last]) continue;
      const int64_t len_a = (a.box.hi[last] - a.box.lo[last]) * t.esize;
      const int64_t len_b = (b.box.hi[last] - b.box.lo[last]) * t.esize;
      if (len_a % 16 == 0 && len_b % 16 == 0) continue;
      if (len_a + len_b > INT32_MAX) continue;
      partner[v[k]] = (int64_t)v[k + 1];
      partner[v[k + 1]] = -2 - (int64_t)v[k];
      ++k;  // the next pair starts after piece B
    }
  }
  return partner;
}

// Pairs of regions of one pass (direct or unpack) that form whole destination rows together:
// same tensor and device group in that pass, the same box but for the last dim, where region A
// ends at region B's start; the last dim contiguous on both sources (message blocks always are)
// and the destination, at least two elements of each piece and two rows. Only rows misaligned by
// construction pair up (the destination pitch or piece A's length is not a multiple of 16
// bytes), where the two plain items would each be walked as short rows. Rows of three or more
// pieces pair consecutive pieces two by two; an odd last piece stays plain. partner[A] = B,
// partner[B] = -2 - A, -1 for an unpaired region.
std::vector<int64_t> gather_pairs(const reshard_plan &p, const std::vector<Role> &roles,
                                  const std::vector<Group> &dev_groups, int set) {
  std::vector<int64_t> partner(p.regions.size(), -1);
  if (!RESHARD_GATHER) return partner;
  if (set == kPack) return scatter_pairs(p, roles);
  // the region's destination group in this pass (the unpack pass reads dense message blocks,
  // contiguous along the last dim by construction)
  auto group_of = [&](size_t i) { return set == kDirect ? roles[i].direct : roles[i].unpack; };

  // candidates keyed by (tensor, device group, the box outside the last dim)
  std::map<std::vector<int64_t>, std::vector<size_t>> rows_of;
  for (size_t i = 0; i < p.regions.size(); ++i) {
    const Region &r = p.regions[i];
    const TensorInfo &t = p.tensors[(size_t)r.tensor];
    const int nd = t.ndim, last = nd - 1;
    if (group_of(i) < 0 || nd < 2) continue;
    if (r.box.hi[last] - r.box.lo[last] < 2 || r.box.hi[last - 1] - r.box.lo[last - 1] < 2) continue;
    if (set == kDirect && t.src_view[(size_t)r.src].strides[last] != 1) continue;
    const Group &g = dev_groups[(size_t)group_of(i)];
    if (t.dst_view[(size_t)g.members[0]].strides[last] != 1) continue;
    std::vector<int64_t> key{r.tensor, group_of(i)};
    for (int d = 0; d < last; ++d) {
      key.push_back(r.box.lo[d]);
      key.push_back(r.box.hi[d]);
    }
    rows_of[key].push_back(i);
  }
  for (auto &kv : rows_of) {
    std::vector<size_t> &v = kv.second;
    if (v.size() < 2) continue;
    const TensorInfo &t = p.tensors[(size_t)p.regions[v[0]].tensor];
    const int last = t.ndim - 1;
    std::sort(v.begin(), v.end(), [&](size_t a, size_t b) { return p.regions[a].box.lo[last] < p.regions[b].box.lo[last]; });
    for (size_t k = 0; k + 1 < v.size(); ++k) {
      const Region &a = p.regions[v[k]], &b = p.regions[v[k + 1]];
      if (a.box.hi[last] != b.box.lo[last]) continue;
      const Group &g = dev_groups[(size_t)group_of(v[k])];
      const int64_t dpitch = t.dst_view[(size_t)g.members[0]].strides[last - 1] * t.esize;
      const int64_t len_a = (a.box.hi[last] - a.box.lo[last]) * t.esize;
      if (dpitch % 16 == 0 && len_a % 16 == 0) continue;
      const int64_t row_b = (b.box.hi[last] - a.box.lo[last]) * t.esize;
      if (row_b > INT32_MAX) continue;
      partner[v[k]] = (int64_t)v[k + 1];
      partner[v[k + 1]] = -2 - (int64_t)v[k];
      ++k;  // the next pair starts after piece B
    }
  }
  return partner;
}

// Gather items of the pair (a, b) in pass `set`: the rows dim is the last but one (outer dims
// merge into it while both sources and the destination step uniformly over them, and are walked
// explicitly otherwise), and each item moves about kGatherItemBytes (read + written over all replicas) in a
// multiple of 8 rows, one or more per warp of the CTA that takes it (measured on the (2,4) ->
// (3,) / (3,2) mesh reshards: 16 rows of 2,732 bytes with one replica, 8 with two, against
// 0.78-0.83 of the copy rate for items of about item_bytes of source).
void emit_gather(reshard_plan &p, size_t a, size_t b, const std::vector<Role> &roles, const std::vector<Group> &dev_groups,
                 int64_t item_bytes, int set) {
  const Region &ra = p.regions[a];
  const TensorInfo &t = p.tensors[(size_t)ra.tensor];
  const int nd = t.ndim, last = nd - 1, rd = nd - 2;
  const int32_t dg = set == kDirect ? roles[a].direct : set == kUnpack ? roles[a].unpack : p.workspace_group;
  int64_t ext[kMaxDims];
  for (int d = 0; d < nd; ++d) ext[d] = ra.box.hi[d] - ra.box.lo[d];
  const int64_t len[2] = {ext[last], p.regions[b].box.hi[last] - p.regions[b].box.lo[last]};
  // dense row-major strides of a piece's message block (its region's extents)
  auto dense = [&](int q, int64_t *st) {
    int64_t acc = 1;
    for (int d = nd - 1; d >= 0; --d) {
      st[d] = acc;
      acc *= d == last ? len[q] : ext[d];
    }
  };
  // each piece's source: its source shard (direct, pack), or its dense block of the received
  // message (unpack: at the region's byte offset recv_off); its destination: the replica group's
  // row (direct, unpack), or its dense block of the outgoing message (pack: at send_off)
  int64_t so[2], sst[2][kMaxDims], dof[2], dst_st[2][kMaxDims];
  int32_t sptr[2];
  for (int q = 0; q < 2; ++q) {
    const size_t ri = q ? b : a;
    const Region &r = p.regions[ri];
    if (set == kUnpack) {
      so[q] = roles[ri].recv_off / t.esize;
      dense(q, sst[q]);
      sptr[q] = (int32_t)(p.workspace_ptr + 1);
    } else {
      const RankView &v = region_source(p, r, so[q]);
      for (int d = 0; d < nd; ++d) sst[q][d] = v.strides[d];
      sptr[q] = (int32_t)(t.src_base + r.src);
    }
    if (set == kPack) {
      dof[q] = roles[ri].send_off / t.esize;
      dense(q, dst_st[q]);
    } else {
      const int64_t *ds = region_dest(p, r, dev_groups[(size_t)dg], dof[q]);
      for (int d = 0; d < nd; ++d) dst_st[q][d] = ds[d];
    }
  }
  const int64_t row_b = (len[0] + len[1]) * t.esize;
  const int64_t nrep = set == kPack ? 1 : (int64_t)dev_groups[(size_t)dg].members.size();
  int64_t per = kGatherItemBytes / (row_b * (1 + nrep)) / kGatherRowStep * kGatherRowStep;
  per = std::min(std::max(per, kGatherRowStep), std::max<int64_t>(1, item_bytes / row_b));
  // outer dims merge into the rows dim while both pieces' sources and destinations step
  // uniformly over them (as the plain items' rows do); the rest are walked explicitly
  int64_t rows = ext[rd];
  int k = rd - 1;
  auto uniform = [&](int d) {
    for (int q = 0; q < 2; ++q)
      if (sst[q][d] != rows * sst[q][rd] || dst_st[q][d] != rows * dst_st[q][rd]) return false;
    return true;
  };
  while (k >= 0 && (ext[k] == 1 || uniform(k))) {
    rows *= ext[k];
    --k;
  }
  int64_t idx[kMaxDims] = {0, 0, 0, 0};
  for (;;) {
    int64_t s0[2] = {so[0], so[1]}, d0[2] = {dof[0], dof[1]};
    for (int d = 0; d <= k; ++d)
      for (int q = 0; q < 2; ++q) {
        s0[q] += idx[d] * sst[q][d];
        d0[q] += idx[d] * dst_st[q][d];
      }
    for (int64_t r = 0; r < rows; r += per) {
      GItem g{};
      g.rows = (int32_t)std::min(per, rows - r);
      for (int q = 0; q < 2; ++q) {
        g.src_off[q] = s0[q] + r * sst[q][rd];
        g.src_pitch[q] = sst[q][rd];
        g.dst_off[q] = d0[q] + r * dst_st[q][rd];
        g.dst_pitch[q] = dst_st[q][rd];
        g.run[q] = (int32_t)len[q];
        g.src[q] = sptr[q];
      }
      g.group = dg;
      g.esize = t.esize;
      g.kind = set == kPack ? kScatterRow : kGatherRow;
      p.gitems[set].push_back(g);
    }
    int d = k;
    for (; d >= 0; --d) {
      if (++idx[d] < ext[d]) break;
      idx[d] = 0;
    }
    if (d < 0) break;
  }
}

// Steps 4 and 5: the device group table (the given replica sets plus the send-buffer group) and
// the work items of the three passes, each region as its role says. `dev_groups` are replica
// sets of destination pointer indices within a tensor's run; a role's group indexes them.
int emit_tables(reshard_plan *plan, const std::vector<Role> &roles, const std::vector<Group> &dev_groups) {
  const int64_t Ns = plan->n_src_ptrs, Nd = plan->n_dst_ptrs;
  plan->workspace_ptr = Ns + 2 * Nd;
  const int32_t recv_ptr = (int32_t)(plan->workspace_ptr + 1);
  plan->grp_start.assign(1, 0);
  plan->mem_ptr.clear();
  plan->mem_off.clear();
  plan->max_fanout = 0;
  for (const Group &g : dev_groups) {
    const TensorInfo &t = plan->tensors[(size_t)g.tensor];
    for (int32_t m : g.members) {
      plan->mem_ptr.push_back((int32_t)(Ns + t.dst_base + m));
      plan->mem_off.push_back(t.dst_view[(size_t)m].offset);
    }
    plan->grp_start.push_back((int32_t)plan->mem_ptr.size());
    plan->max_fanout = std::max(plan->max_fanout, (int)g.members.size());
  }
  plan->workspace_group = (int32_t)dev_groups.size();
  plan->mem_ptr.push_back((int32_t)plan->workspace_ptr);
  plan->mem_off.push_back(0);
  plan->grp_start.push_back((int32_t)plan->mem_ptr.size());

  int64_t plan_bytes = 0;
  for (size_t i = 0; i < plan->regions.size(); ++i)
    if (roles[i].direct >= 0 || roles[i].send_off >= 0 || roles[i].unpack >= 0) plan_bytes += region_bytes(*plan, plan->regions[i]);
  int64_t item_bytes = kMaxItemBytes;
  while (item_bytes > kMinItemBytes && plan_bytes / item_bytes < kItemsPerPlan) item_bytes /= 2;
  std::map<SlabSpec, int32_t> slab_ids;
  const std::vector<int64_t> partner = gather_pairs(*plan, roles, dev_groups, kDirect);
  const std::vector<int64_t> partner_u = gather_pairs(*plan, roles, dev_groups, kUnpack);
  const std::vector<int64_t> partner_p = gather_pairs(*plan, roles, dev_groups, kPack);
  for (auto &gv : plan->gitems) gv.clear();
  for (size_t i = 0; i < plan->regions.size(); ++i) {
    const Region &r = plan->regions[i];
    const Role &role = roles[i];
    const TensorInfo &t = plan->tensors[(size_t)r.tensor];
    const int nd = t.ndim;
    const Box &sb = t.src_box[(size_t)r.src];
    const RankView &sv = t.src_view[(size_t)r.src];
    int64_t ext[kMaxDims], ms[kMaxDims];
    int64_t so = sv.offset;
    for (int d = 0; d < nd; ++d) {
      ext[d] = r.box.hi[d] - r.box.lo[d];
      so += (r.box.lo[d] - sb.lo[d]) * sv.strides[d];
    }
    int64_t dd = 1;
    for (int d = nd - 1; d >= 0; --d) {
      ms[d] = dd;
      dd *= ext[d];
    }
    const int32_t sp = (int32_t)(t.src_base + r.src);
    int64_t slo[kMaxDims], sext[kMaxDims], zero[kMaxDims] = {0, 0, 0, 0};
    for (int d = 0; d < nd; ++d) {
      slo[d] = r.box.lo[d] - sb.lo[d];
      sext[d] = sb.hi[d] - sb.lo[d];
    }
    const ReadSide from_src{sp, sv.offset, slo, sext};
    // destination offset and strides of a device group (all members share the strides)
    auto dst_side = [&](int32_t dg, int64_t &dof) -> const int64_t * {
      const Group &g = dev_groups[(size_t)dg];
      const RankView &dv = t.dst_view[(size_t)g.members[0]];
      dof = 0;
      for (int d = 0; d < nd; ++d) dof += (r.box.lo[d] - g.box.lo[d]) * dv.strides[d];
      return dv.strides;
    };
    if (role.direct >= 0) {
      int64_t dof;
      const int64_t *ds = dst_side(role.direct, dof);
      const size_t n0 = plan->items[kDirect].size();
      emit_region(nd, ext, so, sv.strides, from_src, dof, ds, role.direct, t.esize, item_bytes, plan->items[kDirect],
                  plan->titems[kDirect], slab_ids, plan->slabs);
      // a paired region's rows are written by gather items; its plain items stay in the table
      // (flagged) for the passes that walk plain items only
      if (partner[i] != -1)
        for (size_t k = n0; k < plan->items[kDirect].size(); ++k) plan->items[kDirect][k].pad[0] = kGathered;
      if (partner[i] >= 0) emit_gather(*plan, i, (size_t)partner[i], roles, dev_groups, item_bytes, kDirect);
    }
    if (role.send_off >= 0) {
      const int64_t mo = role.send_off / t.esize;
      const size_t n0 = plan->items[kPack].size();
      emit_region(nd, ext, so, sv.strides, from_src, mo, ms, plan->workspace_group, t.esize, item_bytes,
                  plan->items[kPack], plan->titems[kPack], slab_ids, plan->slabs);
      if (partner_p[i] != -1)
        for (size_t k = n0; k < plan->items[kPack].size(); ++k) plan->items[kPack][k].pad[0] = kGathered;
      if (partner_p[i] >= 0) emit_gather(*plan, i, (size_t)partner_p[i], roles, dev_groups, item_bytes, kPack);
    }
    if (role.unpack >= 0) {
      const int64_t mo = role.recv_off / t.esize;
      const ReadSide from_msg{recv_ptr, mo, zero, ext};
      int64_t dof;
      const int64_t *ds = dst_side(role.unpack, dof);
      const size_t n0 = plan->items[kUnpack].size();
      emit_region(nd, ext, mo, ms, from_msg, dof, ds, role.unpack, t.esize, item_bytes, plan->items[kUnpack],
                  plan->titems[kUnpack], slab_ids, plan->slabs);
      if (partner_u[i] != -1)
        for (size_t k = n0; k < plan->items[kUnpack].size(); ++k) plan->items[kUnpack][k].pad[0] = kGathered;
      if (partner_u[i] >= 0) emit_gather(*plan, i, (size_t)partner_u[i], roles, dev_groups, item_bytes, kUnpack);
    }
  }
#if RESHARD_SIZE_ORDER == 1
  // largest items first: the persistent grid deals items round-robin, so CTAs finish together
  for (auto &iv : plan->items)
    std::stable_sort(iv.begin(), iv.end(), [](const Item &a, const Item &b) {
      return (int64_t)a.rows * a.run * a.esize > (int64_t)b.rows * b.run * b.esize;
    });
#elif RESHARD_SIZE_ORDER == 2
  // by destination: items writing neighbouring bytes of one replica group run close together
  for (auto &iv : plan->items)
    std::stable_sort(iv.begin(), iv.end(), [](const Item &a, const Item &b) {
      return a.group != b.group ? a.group < b.group : a.dst_off < b.dst_off;
    });
#endif
  // transposing items grouped by element size: the executor launches one build of its
  // transposing kernel per element size present, each over a contiguous run of the table
  for (auto &tv : plan->titems)
    std::stable_sort(tv.begin(), tv.end(), [](const TItem &a, const TItem &b) { return a.esize < b.esize; });

  // pointer-table entries each pass reads (sources) and writes (destinations)
  for (int set = 0; set < kNumSets; ++set) {
    std::vector<char> s_used((size_t)Ns, 0), d_used((size_t)Nd, 0);
    auto note = [&](int32_t src, int32_t group) {
      if (src < Ns) s_used[(size_t)src] = 1;
      for (int32_t k = plan->grp_start[(size_t)group]; k < plan->grp_start[(size_t)group + 1]; ++k) {
        const int32_t q = plan->mem_ptr[(size_t)k];
        if (q >= Ns && q < Ns + Nd) d_used[(size_t)(q - Ns)] = 1;
      }
    };
    for (const Item &it : plan->items[set]) note(it.src, it.group);
    for (const TItem &it : plan->titems[set]) note(it.src, it.group);
    plan->used_src[set].clear();
    plan->used_dst[set].clear();
    for (int64_t i = 0; i < Ns; ++i)
      if (s_used[(size_t)i]) plan->used_src[set].push_back((int32_t)i);
    for (int64_t i = 0; i < Nd; ++i)
      if (d_used[(size_t)i]) plan->used_dst[set].push_back((int32_t)(Ns + i));
  }

  int64_t global_bytes = 0;
  for (const TensorInfo &t : plan->tensors) {
    int64_t v2 = t.esize;
    for (int d = 0; d < t.ndim; ++d) v2 *= t.shape[d];
    global_bytes += v2;
  }
  reshard_stats_t &st = plan->stats;
  st.n_tensors = (int64_t)plan->tensors.size();
  st.regions = (int64_t)plan->regions.size();
  st.items = (int64_t)(plan->items[kDirect].size() + plan->titems[kDirect].size());
  st.gather_items = (int64_t)(plan->gitems[kDirect].size() + plan->gitems[kPack].size() + plan->gitems[kUnpack].size());
  st.dst_groups = (int64_t)plan->groups.size();
  st.gather_bcast_bytes = 2 * global_bytes;
  st.global_bytes = global_bytes;
  st.rank = plan->rank;
  st.world = plan->world;
  if ((int64_t)(plan->items[kDirect].size() + plan->items[kPack].size() + plan->items[kUnpack].size() +
                plan->titems[kDirect].size() + plan->titems[kPack].size() + plan->titems[kUnpack].size() +
                plan->gitems[kDirect].size() + plan->gitems[kPack].size() + plan->gitems[kUnpack].size()) > INT32_MAX ||
      (int64_t)plan->mem_ptr.size() > INT32_MAX || (int64_t)plan->slabs.size() > INT32_MAX ||
      pointer_table_size(plan) > INT32_MAX) {
    return fail(RESHARD_ERR_UNSUPPORTED, "plan too large (more than 2^31 items, members or pointers)");
  }
  return RESHARD_OK;
}

int build(const reshard_tensor_spec_t *specs, int n, reshard_plan_t **out) {
  if (!out) return fail(RESHARD_ERR_INVALID_ARG, "out is NULL");
  *out = nullptr;
  std::unique_ptr<reshard_plan> owner(new reshard_plan());
  reshard_plan *plan = owner.get();
  int rc = plan_regions(specs, n, plan);
  if (rc) return rc;

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
      r.msg_off_bytes = msg_bytes;
      msg_bytes += align16(region_bytes(*plan, r));
    }

  // every region: direct to its group, packed at its message offset, unpacked from the same
  std::vector<Role> roles(plan->regions.size());
  int64_t bytes_read = 0, bytes_written = 0;
  for (size_t i = 0; i < plan->regions.size(); ++i) {
    const Region &r = plan->regions[i];
    roles[i] = Role{r.group, r.msg_off_bytes, r.group, r.msg_off_bytes};
    const int64_t b = region_bytes(*plan, r);
    bytes_read += b;
    bytes_written += b * (int64_t)plan->groups[(size_t)r.group].members.size();
  }
  if ((rc = emit_tables(plan, roles, plan->groups))) return rc;
  reshard_stats_t &st = plan->stats;
  st.messages = (int64_t)messages.size();
  st.bytes_read = bytes_read;
  st.bytes_written = bytes_written;
  st.wire_bytes = bytes_read;
  st.message_bytes = msg_bytes;
  st.recv_bytes = msg_bytes;
  *out = owner.release();
  set_error("");
  return RESHARD_OK;
}

// The share of a plan that process `rank` runs when the shards are spread over `world`
// processes (multi-GPU form of the method; see reshard_plan_partition in the header).
int partition(const reshard_plan &g, const int32_t *src_owner, const int32_t *dst_owner, int world, int rank,
              int flags, reshard_plan_t **out) {
  *out = nullptr;
  const int64_t Ns = g.n_src_ptrs, Nd = g.n_dst_ptrs;
  {
    Violations v;
    if (g.rank >= 0) v.add(RESHARD_ERR_INVALID_ARG, "the plan is already partitioned");
    if (world < 1) v.add(RESHARD_ERR_INVALID_ARG, "world must be >= 1");
    if (rank < 0 || rank >= world) v.add(RESHARD_ERR_INVALID_ARG, "rank out of range 0..world-1");
    if (flags & ~RESHARD_STRIPED) v.add(RESHARD_ERR_INVALID_ARG, "unknown flags");
    if ((Ns && !src_owner) || (Nd && !dst_owner)) v.add(RESHARD_ERR_INVALID_ARG, "src_owner or dst_owner is NULL");
    if (!v.lines.empty()) return v.report();
    for (int64_t i = 0; i < Ns; ++i)
      if (src_owner[i] < 0 || src_owner[i] >= world) {
        v.add(RESHARD_ERR_INVALID_ARG, "src_owner[" + std::to_string(i) + "] is not a process of the group");
        if (v.lines.size() >= 8) break;
      }
    for (int64_t i = 0; i < Nd; ++i)
      if (dst_owner[i] < 0 || dst_owner[i] >= world) {
        v.add(RESHARD_ERR_INVALID_ARG, "dst_owner[" + std::to_string(i) + "] is not a process of the group");
        if (v.lines.size() >= 16) break;
      }
    if (!v.lines.empty()) return v.report();
  }
  std::unique_ptr<reshard_plan> owner(new reshard_plan());
  reshard_plan *plan = owner.get();
  plan->tensors = g.tensors;
  plan->groups = g.groups;
  plan->n_src_ptrs = Ns;
  plan->n_dst_ptrs = Nd;
  plan->quant_ok = g.quant_ok;
  plan->quant_why = g.quant_why;
  plan->rank = rank;
  plan->world = world;
  const bool striped = (flags & RESHARD_STRIPED) != 0;

  // source choice and message key of every region of the unpartitioned plan
  typedef std::pair<int32_t, std::vector<int32_t>> MsgKey;  // (sender, other receivers, sorted)
  struct Placed {
    Region r;
    int32_t sender;
    std::vector<int32_t> recv;   // processes other than the sender holding a member
    std::vector<int32_t> local;  // members held by `rank`
  };
  std::vector<Placed> placed;
  placed.reserve(g.regions.size());
  // holders of every source replica group, per tensor: rep pointer index -> holders (ascending)
  std::vector<std::vector<std::vector<int32_t>>> holders(g.tensors.size());
  for (size_t ti = 0; ti < g.tensors.size(); ++ti) {
    const TensorInfo &t = g.tensors[ti];
    holders[ti].resize((size_t)t.n_src);
    for (int64_t p = 0; p < t.n_src; ++p)
      if (t.src_rep[(size_t)p] >= 0) holders[ti][(size_t)t.src_rep[(size_t)p]].push_back((int32_t)p);
  }
  for (size_t i = 0; i < g.regions.size(); ++i) {
    const Region &r = g.regions[i];
    const TensorInfo &t = g.tensors[(size_t)r.tensor];
    const Group &grp = g.groups[(size_t)r.group];
    std::vector<int32_t> procs;
    Placed pl;
    for (int32_t m : grp.members) {
      const int32_t q = dst_owner[t.dst_base + m];
      procs.push_back(q);
      if (q == rank) pl.local.push_back(m);
    }
    std::sort(procs.begin(), procs.end());
    procs.erase(std::unique(procs.begin(), procs.end()), procs.end());
    // holders of the region's source box: a holder on a receiving process keeps that copy local
    const std::vector<int32_t> &hold = holders[(size_t)r.tensor][(size_t)r.src];
    int32_t pick = -1;
    for (int32_t h : hold)
      if (std::binary_search(procs.begin(), procs.end(), src_owner[t.src_base + h])) {
        pick = h;
        break;
      }
    if (pick < 0) pick = hold[i % hold.size()];
    pl.r = r;
    pl.r.src = pick;
    pl.sender = src_owner[t.src_base + pick];
    for (int32_t q : procs)
      if (q != pl.sender) pl.recv.push_back(q);
    placed.push_back(std::move(pl));
  }

  // messages: (sender, receivers) -> regions in plan order, each 16-byte aligned
  std::map<MsgKey, std::vector<size_t>> msgs;
  for (size_t i = 0; i < placed.size(); ++i)
    if (!placed[i].recv.empty()) msgs[MsgKey(placed[i].sender, placed[i].recv)].push_back(i);
  std::vector<int64_t> in_msg(placed.size(), -1);
  std::map<MsgKey, int64_t> msg_size;
  for (auto &kv : msgs) {
    int64_t off = 0;
    for (size_t i : kv.second) {
      in_msg[i] = off;
      off += align16(region_bytes(g, placed[i].r));
    }
    msg_size[kv.first] = off;
  }
  // buffer layouts: every process's send and receive offsets of every message it takes part in
  std::map<std::pair<int32_t, MsgKey>, int64_t> send_at, recv_at;
  std::vector<int64_t> send_end((size_t)world, 0), recv_end((size_t)world, 0);
  for (auto &kv : msg_size) {
    const MsgKey &k = kv.first;
    send_at[std::make_pair(k.first, k)] = send_end[(size_t)k.first];
    send_end[(size_t)k.first] += kv.second;
    for (int32_t q : k.second) {
      recv_at[std::make_pair(q, k)] = recv_end[(size_t)q];
      recv_end[(size_t)q] += kv.second;
    }
  }

  // roles of this rank's regions; device groups are the members this rank holds
  std::map<std::pair<int32_t, std::vector<int32_t>>, int32_t> dev_of;  // (semantic group, local members)
  std::vector<Group> dev_groups;
  auto dev_group = [&](const Placed &p) -> int32_t {
    auto key = std::make_pair(p.r.group, p.local);
    auto f = dev_of.find(key);
    if (f != dev_of.end()) return f->second;
    Group dg;
    dg.tensor = p.r.tensor;
    dg.box = g.groups[(size_t)p.r.group].box;
    dg.members = p.local;
    dev_groups.push_back(dg);
    return dev_of[key] = (int32_t)dev_groups.size() - 1;
  };
  std::vector<Role> roles;
  int64_t bytes_read = 0, bytes_written = 0, local_bytes = 0;
  for (size_t i = 0; i < placed.size(); ++i) {
    const Placed &p = placed[i];
    Role role;
    const int64_t b = region_bytes(g, p.r);
    if (p.sender == rank && !p.local.empty()) {
      role.direct = dev_group(p);
      local_bytes += b;
      bytes_read += b;
      bytes_written += b * (int64_t)p.local.size();
    }
    if (!p.recv.empty()) {
      const MsgKey k(p.sender, p.recv);
      if (p.sender == rank) {
        role.send_off = send_at[std::make_pair(rank, k)] + in_msg[i];
        bytes_read += b;
      }
      if (std::binary_search(p.recv.begin(), p.recv.end(), rank)) {
        role.unpack = dev_group(p);
        role.recv_off = recv_at[std::make_pair(rank, k)] + in_msg[i];
        bytes_written += b * (int64_t)p.local.size();
      }
    }
    if (role.direct < 0 && role.send_off < 0 && role.unpack < 0) continue;
    plan->regions.push_back(p.r);
    roles.push_back(role);
  }

  // transfers, enumerated once for the whole group in message order, kept where `rank` takes part
  int64_t sent = 0, forwarded = 0;
  std::vector<Transfer> phase2;
  for (auto &kv : msg_size) {
    const MsgKey &k = kv.first;
    const int64_t size = kv.second;
    const int32_t s = k.first;
    const std::vector<int32_t> &rv = k.second;
    const int64_t R = (int64_t)rv.size();
    const int64_t s_off = send_at[std::make_pair(s, k)];
    if (!striped || R == 1) {
      for (int32_t q : rv) {
        const int64_t q_off = recv_at[std::make_pair(q, k)];
        if (s == rank) {
          plan->transfers.push_back(Transfer{q, RESHARD_SEND, RESHARD_SEND_BUF, 1, s_off, size});
          sent += size;
        }
        if (q == rank) plan->transfers.push_back(Transfer{s, RESHARD_RECV, RESHARD_RECV_BUF, 1, q_off, size});
      }
      continue;
    }
    std::vector<int64_t> cut((size_t)R + 1);
    for (int64_t j = 0; j <= R; ++j) cut[(size_t)j] = j == R ? size : (size * j / R) / 16 * 16;
    for (int64_t j = 0; j < R; ++j) {
      const int64_t lo = cut[(size_t)j], len = cut[(size_t)j + 1] - lo;
      if (len <= 0) continue;
      const int32_t qk = rv[(size_t)j];
      const int64_t qk_off = recv_at[std::make_pair(qk, k)];
      if (s == rank) {
        plan->transfers.push_back(Transfer{qk, RESHARD_SEND, RESHARD_SEND_BUF, 1, s_off + lo, len});
        sent += len;
      }
      if (qk == rank) plan->transfers.push_back(Transfer{s, RESHARD_RECV, RESHARD_RECV_BUF, 1, qk_off + lo, len});
      for (int32_t qj : rv) {
        if (qj == qk) continue;
        const int64_t qj_off = recv_at[std::make_pair(qj, k)];
        if (qk == rank) {
          phase2.push_back(Transfer{qj, RESHARD_SEND, RESHARD_RECV_BUF, 2, qk_off + lo, len});
          forwarded += len;
        }
        if (qj == rank) phase2.push_back(Transfer{qk, RESHARD_RECV, RESHARD_RECV_BUF, 2, qj_off + lo, len});
      }
    }
  }
  plan->transfers.insert(plan->transfers.end(), phase2.begin(), phase2.end());

  int rc = emit_tables(plan, roles, dev_groups);
  if (rc) return rc;
  reshard_stats_t &st = plan->stats;
  int64_t n_msgs = 0;
  for (auto &kv : msg_size)
    if (kv.first.first == rank || std::binary_search(kv.first.second.begin(), kv.first.second.end(), rank)) ++n_msgs;
  st.messages = n_msgs;
  st.bytes_read = bytes_read;
  st.bytes_written = bytes_written;
  st.wire_bytes = sent + forwarded;
  st.message_bytes = send_end[(size_t)rank];
  st.recv_bytes = recv_end[(size_t)rank];
  st.transfers = (int64_t)plan->transfers.size();
  st.sent_bytes = sent;
  st.forwarded_bytes = forwarded;
  st.local_bytes = local_bytes;
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

extern "C" int reshard_plan_partition(const reshard_plan_t *plan, const int32_t *src_owner, const int32_t *dst_owner,
                                      int world, int rank, int flags, reshard_plan_t **out) {
  if (!out) return fail(RESHARD_ERR_INVALID_ARG, "out is NULL");
  *out = nullptr;
  if (!plan) return fail(RESHARD_ERR_INVALID_ARG, "plan is NULL");
  try {
    return partition(*plan, src_owner, dst_owner, world, rank, flags, out);
  } catch (const std::bad_alloc &) {
    return fail(RESHARD_ERR_OOM, "host allocation failed while partitioning");
  }
}

extern "C" int reshard_plan_transfers(const reshard_plan_t *plan, int phase, int64_t cap, reshard_transfer_t *out,
                                      int64_t *n_out) {
  if (!plan) return fail(RESHARD_ERR_INVALID_ARG, "plan is NULL");
  if (phase != 1 && phase != 2) return fail(RESHARD_ERR_INVALID_ARG, "phase must be 1 or 2");
  int64_t n = 0;
  for (const Transfer &t : plan->transfers) {
    if (t.phase != phase) continue;
    if (out && n < cap) out[n] = reshard_transfer_t{t.peer, t.dir, t.buf, t.phase, t.offset, t.bytes};
    ++n;
  }
  if (n_out) *n_out = n;
  return RESHARD_OK;
}

extern "C" int reshard_plan_stats(const reshard_plan_t *plan, reshard_stats_t *out) {
  if (!plan || !out) return fail(RESHARD_ERR_INVALID_ARG, "plan or out is NULL");
  *out = plan->stats;
  out->last_launches = plan->last_launches;
  out->last_aligned_items = plan->last_aligned;
  out->last_general_items = plan->last_general;
  out->last_rows_kernel = plan->last_rows_kernel;
  out->last_staged_items = plan->last_staged;
  out->last_gather_items = plan->last_gather;
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
  if (set < 0 || set >= 3 * kNumSets) return fail(RESHARD_ERR_INVALID_ARG, "set must be in 0..8");
  static_assert(sizeof(Item) == sizeof(TItem), "both item kinds are 64 bytes");
  size_t count, size = sizeof(Item);
  const void *data;
  if (set < kNumSets) {
    count = plan->items[set].size();
    data = plan->items[set].data();
  } else if (set < 2 * kNumSets) {
    count = plan->titems[set - kNumSets].size();
    data = plan->titems[set - kNumSets].data();
  } else {
    count = plan->gitems[set - 2 * kNumSets].size();
    data = plan->gitems[set - 2 * kNumSets].data();
    size = sizeof(GItem);
  }
  if (n_out) *n_out = (int64_t)count;
  if (items && cap > 0) std::memcpy(items, data, (size_t)std::min<int64_t>(cap, (int64_t)count) * size);
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
