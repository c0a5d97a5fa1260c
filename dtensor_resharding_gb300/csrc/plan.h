// Internal plan representation shared by the host planner (plan.cpp) and the device executor
// (execute.cu). Not part of the public ABI (include/reshard.h).
#pragma once

#include <cstdint>
#include <string>
#include <utility>
#include <vector>

#include "../../include/reshard.h"

namespace reshard {

constexpr int kMaxDims = RESHARD_MAX_DIMS;

// Source bytes per device work item. Regions are cut into items of about this size so a
// persistent grid that walks the item table round-robin stays balanced: the largest power of
// two in [kMinItemBytes, kMaxItemBytes] that still gives about kItemsPerPlan items per plan
// (small plans get small items, so every SM has work).
#ifndef RESHARD_ITEMS_PER_PLAN
#define RESHARD_ITEMS_PER_PLAN 512
#endif
#ifndef RESHARD_MIN_ITEM_KIB
#define RESHARD_MIN_ITEM_KIB 64
#endif
constexpr int64_t kMaxItemBytes = 256 * 1024;
constexpr int64_t kMinItemBytes = RESHARD_MIN_ITEM_KIB * 1024;
constexpr int64_t kItemsPerPlan = RESHARD_ITEMS_PER_PLAN;
// Long runs are cut at multiples of this many elements (keeps MXFP8 blocks whole).
constexpr int64_t kRunSplitElems = 2048;

// Half-open box [lo, hi) per tensor dim.
struct Box {
  int64_t lo[kMaxDims];
  int64_t hi[kMaxDims];
};

// A rank's local shard inside its buffer (elements).
struct RankView {
  int64_t offset = 0;
  int64_t strides[kMaxDims] = {0, 0, 0, 0};
  bool dense = true;  // strides were not given (dense row-major of the local shape)
};

// Device work item: `rows` rows of `run` contiguous elements. Row i of the source starts at
// element src_off + i * src_pitch of pointer `src`; row i of destination replica m starts at
// element member_offset[m] + dst_off + i * dst_pitch of that member's pointer.
struct alignas(16) Item {
  int64_t src_off;
  int64_t dst_off;
  int64_t src_pitch;
  int64_t dst_pitch;
  int32_t rows;
  int32_t run;
  int32_t src;    // pointer-table index of the source buffer
  int32_t group;  // destination group (replica set) index
  int32_t esize;  // bytes per element of the tensor
  int32_t pad[3];
};
static_assert(sizeof(Item) == 64, "work item is one 64-byte descriptor");

// Transposing work item: the source is contiguous along the item's columns (C), the
// destination along its rows (R). Element (r, c) is read at src_off + r * src_pitch + c of
// pointer `src` and written at member_offset + dst_off + c * dst_pitch + r of every member of
// `group`. `map` names the source slab (a 2-D tensor map encoded at execute time); (x, y) are
// the item's (c0, r0) coordinates in that slab.
struct alignas(16) TItem {
  int64_t src_off;
  int64_t dst_off;
  int64_t src_pitch;
  int64_t dst_pitch;
  int32_t rows;
  int32_t cols;
  int32_t src;
  int32_t group;
  int32_t esize;
  int32_t map;
  int32_t x;
  int32_t y;
};
static_assert(sizeof(TItem) == 64, "transposing item is one 64-byte descriptor");

// Pair direct regions into gather items (0 turns it off: every region is walked as plain items).
#ifndef RESHARD_GATHER
#define RESHARD_GATHER 1
#endif
// Bytes a gather item moves (read + written over all replicas), in rows of a multiple of 8.
#ifndef RESHARD_GATHER_ITEM_KIB
#define RESHARD_GATHER_ITEM_KIB 96
#endif
constexpr int64_t kGatherItemBytes = RESHARD_GATHER_ITEM_KIB * 1024;
constexpr int64_t kGatherRowStep = 8;

// Pair item: `rows` rows of two pieces, walked together by one warp. Row i of piece p is
// run[p] elements read at src_off[p] + i * src_pitch[p] of pointer src[p] and written at
// member_offset[m] + dst_off[p] + i * dst_pitch[p] of every member m of `group`.
//   kGatherRow (direct and unpack passes): one destination row made of two source pieces side by
//     side (dst_off[1] = dst_off[0] + run[0], dst_pitch[1] = dst_pitch[0]); the sources are two
//     source shards in the direct pass, two message blocks of the receive buffer in the unpack
//     pass.
//   kScatterRow (pack pass): one source row split into two message blocks (src[1] = src[0],
//     src_off[1] = src_off[0] + run[0]); the group is the send buffer's.
// A pair item replaces the plain items of its two regions, which stay in the pass's table
// flagged kGathered (the MXFP8 passes and the allocation-free entry point walk the plain items).
constexpr int32_t kGatherRow = 0;
constexpr int32_t kScatterRow = 1;
struct alignas(16) GItem {
  int64_t src_off[2];
  int64_t src_pitch[2];
  int64_t dst_off[2];
  int64_t dst_pitch[2];
  int32_t run[2];
  int32_t src[2];
  int32_t rows;
  int32_t group;
  int32_t esize;
  int32_t kind;
};
static_assert(sizeof(GItem) == 96, "pair item is one 96-byte descriptor");

// A pair item with its addresses resolved for the current pointer table (built on the host
// whenever the table changes, so the kernel follows no pointer table): row 0 of both pieces'
// sources; for a gather row, row 0 in the first two replicas (replicas past the second are looked
// up through the group table, at member_offset * esize + dst_off_b of each member's pointer); for
// a scatter row, row 0 of each piece's destination. Pitches and lengths in bytes.
struct alignas(16) GBound {
  uint64_t src[2];
  uint64_t dst[2];      // gather: replicas 0 and 1 (dst[1] == dst[0] with one); scatter: pieces 0 and 1
  int64_t sp[2];
  int64_t dp[2];        // destination pitch (gather: dp[0]; scatter: per piece)
  int64_t dst_off_b;
  int32_t B;            // piece 0's bytes per row
  int32_t rb;           // bytes per row, both pieces
  int32_t rows;
  int32_t group;
  int32_t nrep;
  int32_t esize;
  int32_t kind;
  int32_t pad;
};
static_assert(sizeof(GBound) == 112, "resolved pair item is one 112-byte descriptor");
// Item.pad[0] flag: the item's rows are written by a gather item instead
constexpr int32_t kGathered = 1;

// A 2-D source slab read by TMA: element (y, x) at base_off + y * pitch + x (elements) of
// pointer `ptr`, extents x < cols, y < rows.
struct SlabSpec {
  int32_t ptr;
  int32_t esize;
  int64_t base_off;
  int64_t cols;
  int64_t rows;
  int64_t pitch;
  bool operator<(const SlabSpec &o) const {
    if (ptr != o.ptr) return ptr < o.ptr;
    if (esize != o.esize) return esize < o.esize;
    if (base_off != o.base_off) return base_off < o.base_off;
    if (cols != o.cols) return cols < o.cols;
    if (rows != o.rows) return rows < o.rows;
    return pitch < o.pitch;
  }
};

// Rows and bytes of one transpose tile (one 128-byte swizzle span per tile row).
constexpr int kTileRows = 128;
constexpr int kTileRowBytes = 128;
// Tiles per transposing item along each dim.
constexpr int kItemTiles = 4;

struct TensorInfo {
  int ndim = 0;
  int64_t shape[kMaxDims] = {1, 1, 1, 1};
  int dtype = 0;
  int esize = 0;
  int64_t n_src = 0, n_dst = 0;        // ranks on each side
  int64_t src_base = 0, dst_base = 0;  // first pointer index of this tensor (flat, per side)
  std::vector<Box> src_box, dst_box;   // per pointer index
  std::vector<RankView> src_view, dst_view;
  // per source pointer index: the lowest pointer index holding the same box (its replica
  // group's representative), or -1 for an empty shard
  std::vector<int32_t> src_rep;
};

struct Region {
  int32_t tensor;
  int32_t src;    // pointer index within the tensor's source run (the chosen holder)
  int32_t group;  // plan-wide destination group id
  Box box;        // global coordinates
  int64_t msg_off_bytes = 0;  // packed-mode workspace offset (16-byte aligned)
};

// How a plan executes one region: `direct` (device group index, or -1) copies the source to
// that group's members; `send_off` (bytes, or -1) packs it into the send buffer; `unpack`
// (device group index, or -1) copies it from the receive buffer at `recv_off` to the group.
struct Role {
  int32_t direct = -1;
  int64_t send_off = -1;
  int32_t unpack = -1;
  int64_t recv_off = -1;
};

// One point-to-point transfer of a partitioned plan (mirrors reshard_transfer_t).
struct Transfer {
  int32_t peer;
  int32_t dir;    // RESHARD_SEND / RESHARD_RECV
  int32_t buf;    // RESHARD_SEND_BUF / RESHARD_RECV_BUF
  int32_t phase;  // 1 or 2
  int64_t offset;
  int64_t bytes;
};

struct Group {
  int32_t tensor;
  std::vector<int32_t> members;  // destination pointer indices within the tensor's run
  Box box;
};

enum ItemSet { kDirect = 0, kPack = 1, kUnpack = 2, kNumSets = 3 };

}  // namespace reshard

struct reshard_plan {
  std::vector<reshard::TensorInfo> tensors;
  std::vector<reshard::Region> regions;
  std::vector<reshard::Group> groups;  // plan-wide; one extra group for the workspace is
                                       // appended in the device tables
  int64_t n_src_ptrs = 0, n_dst_ptrs = 0;
  std::vector<reshard::Item> items[reshard::kNumSets];
  std::vector<reshard::TItem> titems[reshard::kNumSets];  // transposing items of each pass
  std::vector<reshard::GItem> gitems[reshard::kNumSets];   // gather items of each pass (none in pack)
  std::vector<reshard::GBound> gbound[reshard::kNumSets];  // ... resolved for the current pointer table
  std::vector<reshard::SlabSpec> slabs;                    // TMA source slabs (all passes)
  // group table (device layout): members of group g are [grp_start[g], grp_start[g + 1])
  std::vector<int32_t> grp_start;
  std::vector<int32_t> mem_ptr;   // pointer-table index of each member's data pointer
  std::vector<int64_t> mem_off;   // member's view offset (elements)
  int32_t workspace_group = -1;  // device group whose one member is the send buffer
  int64_t workspace_ptr = -1;     // pointer-table index of the send buffer; the receive
                                  // buffer follows it
  int max_fanout = 0;
  reshard_stats_t stats{};
  bool quant_ok = false;
  std::string quant_why;
  // partitioned plans (reshard_plan_partition): the process this plan runs on, or -1
  int rank = -1;
  int world = 0;
  std::vector<reshard::Transfer> transfers;  // phase 1 entries first, then phase 2
  // pointer-table indices of the sources read and the destinations written by each pass
  std::vector<int32_t> used_src[reshard::kNumSets], used_dst[reshard::kNumSets];

  // device state (bound at the first execute)
  int device = -1;
  void *d_items[reshard::kNumSets] = {nullptr, nullptr, nullptr};
  void *d_titems[reshard::kNumSets] = {nullptr, nullptr, nullptr};
  void *d_gbound[reshard::kNumSets] = {nullptr, nullptr, nullptr};  // the resolved gather items
  uint64_t gbound_version[reshard::kNumSets] = {0, 0, 0};           // the pointer-table version of each
  void *d_maps = nullptr;      // one 128-byte CUtensorMap per slab (64-byte aligned)
  int32_t *d_map_ok = nullptr; // 1 where the slab's map could be encoded
  int32_t *d_status = nullptr; // device-side status word (bit 0: a TMA wait timed out)
  // copy items split by alignment for the current pointers: cls_idx[set] lists the items that
  // are 16-byte aligned everywhere first (n_aligned of them), then the misaligned items of many
  // short rows for the bulk-staged kernel (n_staged), then the rest
  std::vector<int32_t> cls_idx[reshard::kNumSets];
  int32_t n_aligned[reshard::kNumSets] = {0, 0, 0};
  int32_t n_staged[reshard::kNumSets] = {0, 0, 0};  // next in cls_idx: the bulk-staged items
  int32_t n_general[reshard::kNumSets] = {0, 0, 0}; // last in cls_idx: the rest (gathered items are left out)
  int32_t *d_cls_idx[reshard::kNumSets] = {nullptr, nullptr, nullptr};
  uint64_t cls_version[reshard::kNumSets] = {0, 0, 0};
  uint64_t ptr_version = 0;  // bumped whenever the pointer table changes
  int64_t last_launches = 0; // kernel launches enqueued by the last execute
  int64_t last_aligned = 0;  // copy items of the last pass that took the aligned walker
  int64_t last_general = 0;  // ... and the general walker
  int64_t last_rows_kernel = 0;  // 1 when those ran in the many-rows build of the general walker
  int64_t last_staged = 0;       // copy items of the last pass run by the bulk-staged kernel
  int64_t last_gather = 0;       // gather items run by the last execute (all its passes)
  bool gen_rows[reshard::kNumSets] = {false, false, false};  // general items mostly short rows
  int32_t *d_grp_start = nullptr;
  int32_t *d_mem_ptr = nullptr;
  int64_t *d_mem_off = nullptr;
  uint64_t *d_ptrs = nullptr;
  void *d_workspace = nullptr;
  std::vector<uint64_t> ptr_cache;  // the pointer table the kernels last saw, caller's values
  std::vector<uint64_t> dev_ptrs;   // ... as the kernels see them (host memory by its device alias)
  std::vector<uint8_t> ptr_host;    // 1 where an entry is page-locked host memory
  bool any_host = false;            // some pointer is page-locked host memory
  bool ptr_cache_valid = false;
  // completion of the last execute on each stream it used (waited for by destroy)
  std::vector<std::pair<void *, void *>> done_events;  // (cudaStream_t, cudaEvent_t)
};

namespace reshard {
void set_error(const std::string &msg);
int fail(int code, const std::string &msg);
int64_t pointer_table_size(const reshard_plan *p);  // Ns + 2 Nd + 2
}  // namespace reshard
