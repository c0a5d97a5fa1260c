// Device executor of the reshard plan: persistent descriptor-walking kernels for sm_103a.
//
// Every item's source rows are read once and written to every destination replica of its group
// (the fan-out of "xferdtensor Transports" in the NeMo-RL design doc "NCCL Reshard Refit
// (Experimental)"). The same walkers serve the direct mode and both halves of the packed mode
// (pack: source -> contiguous message; unpack: message -> destination replicas), the messages a
// wire transport would carry ("NeMo-RL: Optimizing Non-Colocated Refit", "Optimization #2":
// pack into one contiguous buffer).
// - reshard_copy_aligned_kernel: items 16-byte aligned on every side; 16-byte streaming copies,
//   8 loads in flight per thread.
// - reshard_copy_kernel / reshard_copy_rows_kernel: every other item (one warp per row,
//   funnel-shifted 16-byte destination words); two builds of one walker, for long rows and for
//   many short rows.
// - reshard_transpose_kernel: regions whose two sides are contiguous along different dims; TMA
//   box loads into swizzled shared memory, column runs stored from there.
// - reshard_mxfp8_kernel: the copy walk with the receive-side BF16 -> MXFP8 epilogue (design
//   doc, "Enabling It": generation ranks quantize each received BF16 shard), by the OCP MX v1.0
//   rule: per 32 contiguous elements along the destination's last dim, the E8M0 scale
//   X = floor(log2 amax) - 8 and E4M3 elements v / 2^X rounded to nearest even, saturating at
//   448. The two lanes holding a block combine their amax with a warp shuffle.
//
// Nothing here is a contraction; every kernel is bound by HBM bandwidth. Sources and
// destinations must not overlap in memory.
#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_runtime.h>

#include <algorithm>
#include <cstdio>
#include <cstring>
#include <mutex>
#include <string>
#include <utility>

#include "plan.h"

namespace reshard {

// Launch shape; the defaults are the measured best on GB300 (build-time overridable for sweeps).
#ifndef RESHARD_BLOCK
#define RESHARD_BLOCK 256
#endif
#ifndef RESHARD_UNROLL
#define RESHARD_UNROLL 8
#endif
#ifndef RESHARD_MIN_BLOCKS
#define RESHARD_MIN_BLOCKS 2
#endif
#ifndef RESHARD_GEN_MIN_BLOCKS
#define RESHARD_GEN_MIN_BLOCKS 4
#endif
#ifndef RESHARD_GEN_UNROLL
#define RESHARD_GEN_UNROLL 2
#endif
#ifndef RESHARD_ROWS_MIN_BLOCKS
#define RESHARD_ROWS_MIN_BLOCKS 6
#endif
#ifndef RESHARD_ROWS_GEN_UNROLL
#define RESHARD_ROWS_GEN_UNROLL 1
#endif
#ifndef RESHARD_ROWS_MAX_RUN
#define RESHARD_ROWS_MAX_RUN 4096
#endif
constexpr int kBlock = RESHARD_BLOCK;    // threads per CTA
constexpr int kUnroll = RESHARD_UNROLL;        // 16-byte loads in flight per thread (aligned walker)
constexpr int kGenUnroll = RESHARD_GEN_UNROLL;  // the same in the general walker's aligned path
constexpr int kMaxFan = 8;               // destination replicas held in registers per pass
#ifndef RESHARD_GEN_SMEM_ITEM
#define RESHARD_GEN_SMEM_ITEM 1
#endif
#ifndef RESHARD_GEN_FAN
#define RESHARD_GEN_FAN 8
#endif
constexpr int kGenFan = RESHARD_GEN_FAN;  // the same in the general walker

// Programmatic dependent launch: every launch of this file may start its CTAs while the grid
// before it on the stream drains (they occupy SM slots as that grid's CTAs retire), and every
// kernel's first act is griddepcontrol.wait, which returns only once the grids it depends on
// have completed and their writes are visible: stream order is unchanged, only the launch
// latency is hidden.
#ifndef RESHARD_PDL
#define RESHARD_PDL 1
#endif
#ifndef RESHARD_GEN_OVERLAP
#define RESHARD_GEN_OVERLAP RESHARD_PDL
#endif
__device__ __forceinline__ void pdl_enter() {
#if RESHARD_PDL
  asm volatile("griddepcontrol.wait;" ::: "memory");
#endif
}

// Called by a CTA as it starts its last item (and by a CTA with none): once every CTA of the
// grid has called it, the next launch on the stream may be scheduled. Not earlier, so that its
// waiting CTAs never take SM slots ahead of this grid's own.
__device__ __forceinline__ void pdl_last_item(int k, int n_items) {
#if RESHARD_PDL
  if (k + (int)gridDim.x >= n_items) asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
#endif
}

// ------------------------------------------------------------------------------ helpers --

#ifndef RESHARD_LOAD_HINT
#define RESHARD_LOAD_HINT 0
#endif
#ifndef RESHARD_STORE_HINT
#define RESHARD_STORE_HINT 0
#endif

// Streaming 16-byte load: each source byte is read once per launch.
__device__ __forceinline__ uint4 load_stream(const uint8_t *p) {
#if RESHARD_LOAD_HINT == 0
  return __ldcs(reinterpret_cast<const uint4 *>(p));
#elif RESHARD_LOAD_HINT == 1
  return __ldg(reinterpret_cast<const uint4 *>(p));
#else
  uint4 v;
  asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0,%1,%2,%3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w) : "l"(p));
  return v;
#endif
}

#ifndef RESHARD_WIDE
#define RESHARD_WIDE 0
#endif

// 32-byte global load / store (sm_100 and later accept 256-bit vectors on global memory).
__device__ __forceinline__ void load_stream32(const uint8_t *p, uint4 &a, uint4 &b) {
  asm volatile("ld.global.nc.L1::no_allocate.v8.b32 {%0,%1,%2,%3,%4,%5,%6,%7}, [%8];"
               : "=r"(a.x), "=r"(a.y), "=r"(a.z), "=r"(a.w), "=r"(b.x), "=r"(b.y), "=r"(b.z), "=r"(b.w)
               : "l"(p));
}

__device__ __forceinline__ void store_stream32(uint8_t *p, uint4 a, uint4 b) {
  asm volatile("st.global.cs.v8.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8};"
               :
               : "l"(p), "r"(a.x), "r"(a.y), "r"(a.z), "r"(a.w), "r"(b.x), "r"(b.y), "r"(b.z), "r"(b.w)
               : "memory");
}

// Streaming 16-byte store: destinations are not read back by this launch.
__device__ __forceinline__ void store_stream(uint8_t *p, uint4 v) {
#if RESHARD_STORE_HINT == 0
  __stcs(reinterpret_cast<uint4 *>(p), v);
#else
  *reinterpret_cast<uint4 *>(p) = v;
#endif
}

// Bytes [sh, sh + 16) of the 32-byte concatenation lo:hi (little endian), sh in [0, 16).
__device__ __forceinline__ uint4 shift_bytes(uint4 lo, uint4 hi, int sh) {
  const int r = (sh & 3) * 8;
  uint32_t x0, x1, x2, x3, x4;
  switch (sh >> 2) {
    case 0: x0 = lo.x; x1 = lo.y; x2 = lo.z; x3 = lo.w; x4 = hi.x; break;
    case 1: x0 = lo.y; x1 = lo.z; x2 = lo.w; x3 = hi.x; x4 = hi.y; break;
    case 2: x0 = lo.z; x1 = lo.w; x2 = hi.x; x3 = hi.y; x4 = hi.z; break;
    default: x0 = lo.w; x1 = hi.x; x2 = hi.y; x3 = hi.z; x4 = hi.w; break;
  }
  uint4 o;
  o.x = __funnelshift_r(x0, x1, r);
  o.y = __funnelshift_r(x1, x2, r);
  o.z = __funnelshift_r(x2, x3, r);
  o.w = __funnelshift_r(x3, x4, r);
  return o;
}

// Bytes [kmin, kmax) of the 16-byte word `o` into the 16-byte aligned `word`, each piece the
// widest naturally aligned store that fits (at most 7 stores instead of up to 15 bytes).
__device__ __forceinline__ void store_partial(uint8_t *word, uint4 o, int kmin, int kmax) {
  int k = kmin;
  while (k < kmax) {
    const int left = kmax - k;
    const uint32_t w = k < 4 ? o.x : k < 8 ? o.y : k < 12 ? o.z : o.w;
    if ((k & 7) == 0 && left >= 8) {
      *reinterpret_cast<uint2 *>(word + k) = k == 0 ? make_uint2(o.x, o.y) : make_uint2(o.z, o.w);
      k += 8;
    } else if ((k & 3) == 0 && left >= 4) {
      *reinterpret_cast<uint32_t *>(word + k) = w;
      k += 4;
    } else if ((k & 1) == 0 && left >= 2) {
      *reinterpret_cast<uint16_t *>(word + k) = (uint16_t)(w >> ((k & 2) * 8));
      k += 2;
    } else {
      word[k] = (uint8_t)(w >> ((k & 3) * 8));
      k += 1;
    }
  }
}

// ------------------------------------------------------------------- copy with fan-out --

// Every source, destination, run and pitch 16-byte aligned: straight 16-byte copies.
template <int U, int NF>
__device__ __forceinline__ void copy_aligned(const uint8_t *__restrict__ src, uint8_t *const *dst, int nf, int rows,
                                             int64_t run_b, int64_t sp_b, int64_t dp_b) {
  const int nw = (int)(run_b >> 4);
  const int total = rows * nw;
  // word j is (row j / nw, word j % nw); consecutive slots of a thread are kBlock apart and its
  // passes kBlock * U apart, so (row, word) step by quotients and remainders taken once
  const int q_blk = kBlock / nw, r_blk = kBlock - q_blk * nw;
  const int q_pass = (kBlock * U) / nw, r_pass = kBlock * U - q_pass * nw;
  int row0 = (int)threadIdx.x / nw, col0 = (int)threadIdx.x - row0 * nw;
  for (int base = threadIdx.x; base < total; base += kBlock * U) {
    uint4 v[U];
    int64_t doff[U];
    int r = row0, w = col0;
#pragma unroll
    for (int u = 0; u < U; ++u) {
      const int j = base + u * kBlock;
      if (j < total) {
        v[u] = load_stream(src + r * sp_b + 16 * (int64_t)w);
        doff[u] = r * dp_b + 16 * (int64_t)w;
      }
      w += r_blk;
      r += q_blk;
      if (w >= nw) {
        w -= nw;
        ++r;
      }
    }
    col0 += r_pass;
    row0 += q_pass;
    if (col0 >= nw) {
      col0 -= nw;
      ++row0;
    }
#pragma unroll
    for (int u = 0; u < U; ++u) {
      if (base + u * kBlock < total) {
#pragma unroll
        for (int f = 0; f < NF; ++f)
          if (f < nf) store_stream(dst[f] + doff[u], v[u]);
      }
    }
  }
}

// Every source, destination, run and pitch 32-byte aligned: 32-byte copies.
template <int NF>
__device__ __forceinline__ void copy_aligned32(const uint8_t *__restrict__ src, uint8_t *const *dst, int nf, int rows,
                                               int64_t run_b, int64_t sp_b, int64_t dp_b) {
  const int nw = (int)(run_b >> 5);
  const int total = rows * nw;
  for (int base = threadIdx.x; base < total; base += kBlock * kUnroll) {
    uint4 va[kUnroll], vb[kUnroll];
    int64_t doff[kUnroll];
#pragma unroll
    for (int u = 0; u < kUnroll; ++u) {
      const int j = base + u * kBlock;
      if (j < total) {
        const int r = rows == 1 ? 0 : j / nw;
        const int w = j - r * nw;
        load_stream32(src + r * sp_b + 32 * (int64_t)w, va[u], vb[u]);
        doff[u] = r * dp_b + 32 * (int64_t)w;
      }
    }
#pragma unroll
    for (int u = 0; u < kUnroll; ++u) {
      if (base + u * kBlock < total) {
#pragma unroll
        for (int f = 0; f < NF; ++f)
          if (f < nf) store_stream32(dst[f] + doff[u], va[u], vb[u]);
      }
    }
  }
}

// The same funnel-shift copy with one warp per row: the row's destination misalignment, its
// source phase and hence the shift are computed once per row, the lanes walk the row's
// destination words, and the shift amount is warp-uniform. Word w of a row holds row bytes
// [16 w - a, 16 w - a + 16), a the row's destination misalignment. A single-row item is cut
// into virtual rows of kVRow bytes whose boundaries fall on destination 16-byte boundaries, so
// that no destination word is shared by two rows.
#ifndef RESHARD_ROW_UNROLL
#define RESHARD_ROW_UNROLL 2
#endif
#ifndef RESHARD_VROW_PASSES
#define RESHARD_VROW_PASSES 2
#endif
#ifndef RESHARD_GEN_ROW_UNROLL
#define RESHARD_GEN_ROW_UNROLL 3
#endif

// RU: destination words per lane in flight; a virtual row is RESHARD_VROW_PASSES passes long.
template <int NF, int RU>
__device__ __forceinline__ void copy_shifted_rows(const uint8_t *__restrict__ src, uint8_t *const *dst, int nf,
                                                  int rows, int64_t run_b, int64_t sp_b, int64_t dp_b) {
  constexpr int kVRow = 32 * 16 * RU * RESHARD_VROW_PASSES;  // bytes per virtual row
  const int lane = threadIdx.x & 31;
  const uintptr_t d0 = reinterpret_cast<uintptr_t>(dst[0]);
  const int a0 = (int)(d0 & 15);
  const bool split = rows == 1;
  const int nrow = split ? (int)((run_b + a0 + kVRow - 1) / kVRow) : rows;
  for (int r = threadIdx.x >> 5; r < nrow; r += kBlock / 32) {
    int64_t sb, db, rb;  // source and destination byte offset of the row, its length
    if (split) {
      sb = r ? (int64_t)r * kVRow - a0 : 0;
      const int64_t e = (int64_t)(r + 1) * kVRow - a0;
      rb = (e < run_b ? e : run_b) - sb;
      db = sb;
    } else {
      sb = r * sp_b;
      db = r * dp_b;
      rb = run_b;
    }
    const int a = (int)((d0 + db) & 15);
    const int nw = (int)((a + rb + 15) >> 4);  // destination words the row touches
    const uintptr_t p00 = reinterpret_cast<uintptr_t>(src) + sb - a;  // source of word 0's byte 0
    const int sh = (int)(p00 & 15);
    const uint8_t *blk0 = reinterpret_cast<const uint8_t *>(p00 - sh);
    const int64_t dbase = db - a;  // destination offset of word 0's byte 0
    for (int w0 = lane; w0 < nw; w0 += 32 * RU) {
      uint4 lo[RU], hi[RU];
      int kmin[RU], kmax[RU];
#pragma unroll
      for (int u = 0; u < RU; ++u) {
        const int w = w0 + 32 * u;
        kmin[u] = 16;
        kmax[u] = 0;
        lo[u] = make_uint4(0, 0, 0, 0);
        hi[u] = make_uint4(0, 0, 0, 0);
        if (w < nw) {
          const int64_t start = 16 * (int64_t)w - a;
          kmin[u] = w == 0 ? a : 0;
          kmax[u] = rb - start < 16 ? (int)(rb - start) : 16;
          const uint8_t *blk = blk0 + 16 * (int64_t)w;
          if (kmin[u] < 16 - sh) lo[u] = __ldg(reinterpret_cast<const uint4 *>(blk));
          if (sh && kmax[u] > 16 - sh) hi[u] = __ldg(reinterpret_cast<const uint4 *>(blk + 16));
        }
      }
#pragma unroll
      for (int u = 0; u < RU; ++u) {
        if (kmin[u] >= kmax[u]) continue;
        const uint4 o = sh ? shift_bytes(lo[u], hi[u], sh) : lo[u];
        const int64_t dpos = dbase + 16 * (int64_t)(w0 + 32 * u);
        if (kmin[u] == 0 && kmax[u] == 16) {
#pragma unroll
          for (int f = 0; f < NF; ++f)
            if (f < nf) store_stream(dst[f] + dpos, o);
        } else {
#pragma unroll
          for (int f = 0; f < NF; ++f)
            if (f < nf) store_partial(dst[f] + dpos, o, kmin[u], kmax[u]);
        }
      }
    }
  }
}

// dst[f] for a runtime f without indexing the array (keeps it in registers).
template <int NF>
__device__ __forceinline__ uint8_t *pick(uint8_t *const *dst, int f) {
  uint8_t *p = dst[0];
#pragma unroll
  for (int g = 1; g < NF; ++g) p = f == g ? dst[g] : p;
  return p;
}

// Resolve item k of a launch: items[idx[k]] when an index list is given, else items[k].
__device__ __forceinline__ int item_index(const int32_t *idx, int k) { return idx ? idx[k] : k; }

// The general walker: aligned, 32-byte-aligned and funnel-shift paths, any item. GU is the
// unroll of its aligned path (which serves items found misaligned after all, and every item of
// the allocation-free entry point).
template <int GU, int RU>
__device__ __forceinline__ void general_walk(const Item *__restrict__ items, const int32_t *__restrict__ idx,
                                             int n_items, const uint64_t *__restrict__ ptrs,
                                             const int32_t *__restrict__ gstart, const int32_t *__restrict__ mptr,
                                             const int64_t *__restrict__ moff) {
#if RESHARD_GEN_SMEM_ITEM
  // item descriptors double-buffered in shared memory: 16 threads fetch the next one while the
  // current one is copied, so no thread holds a prefetched descriptor in registers
  __shared__ Item s_item[2];
  constexpr int kWords = (int)(sizeof(Item) / sizeof(uint32_t));
  if (threadIdx.x < kWords && blockIdx.x < n_items)
    reinterpret_cast<uint32_t *>(&s_item[0])[threadIdx.x] =
        __ldg(reinterpret_cast<const uint32_t *>(items + item_index(idx, blockIdx.x)) + threadIdx.x);
  __syncthreads();
  int buf = 0;
  for (int k = blockIdx.x; k < n_items; k += gridDim.x, buf ^= 1) {
    pdl_last_item(k, n_items);
    if (threadIdx.x < kWords && k + (int)gridDim.x < n_items)
      reinterpret_cast<uint32_t *>(&s_item[buf ^ 1])[threadIdx.x] =
          __ldg(reinterpret_cast<const uint32_t *>(items + item_index(idx, k + gridDim.x)) + threadIdx.x);
    const Item &it = s_item[buf];
#else
  Item nxt;
  if (blockIdx.x < n_items) nxt = items[item_index(idx, blockIdx.x)];
  for (int k = blockIdx.x; k < n_items; k += gridDim.x) {
    pdl_last_item(k, n_items);
    const Item it = nxt;
    // the next item's descriptor is in flight while this one is copied
    if (k + (int)gridDim.x < n_items) nxt = items[item_index(idx, k + gridDim.x)];
#endif
    const int64_t es = it.esize;
    const uint8_t *src = reinterpret_cast<const uint8_t *>(ptrs[it.src]) + it.src_off * es;
    const int g0 = gstart[it.group];
    const int nrep = gstart[it.group + 1] - g0;
    const int64_t run_b = (int64_t)it.run * es;
    const int64_t sp_b = it.src_pitch * es, dp_b = it.dst_pitch * es;
    const uintptr_t geo = reinterpret_cast<uintptr_t>(src) | (uintptr_t)run_b |
                          (it.rows > 1 ? (uintptr_t)(sp_b | dp_b) : 0);
    for (int f0 = 0; f0 < nrep; f0 += kGenFan) {
      const int nf = min(kGenFan, nrep - f0);
      uint8_t *dst[kGenFan];
      uintptr_t amask = geo;
      bool same = true;
#pragma unroll
      for (int f = 0; f < kGenFan; ++f) {
        dst[f] = nullptr;
        if (f < nf) {
          const int m = g0 + f0 + f;
          dst[f] = reinterpret_cast<uint8_t *>(ptrs[mptr[m]]) + (moff[m] + it.dst_off) * es;
          amask |= reinterpret_cast<uintptr_t>(dst[f]);
          same = same && (((reinterpret_cast<uintptr_t>(dst[f]) ^ reinterpret_cast<uintptr_t>(dst[0])) & 15) == 0);
        }
      }
      if (RESHARD_WIDE && (amask & 31) == 0) {
        copy_aligned32<kGenFan>(src, dst, nf, it.rows, run_b, sp_b, dp_b);
      } else if ((amask & 15) == 0) {
        copy_aligned<GU, kGenFan>(src, dst, nf, it.rows, run_b, sp_b, dp_b);
      } else if (same && nf <= 2) {
        copy_shifted_rows<2, RU>(src, dst, nf, it.rows, run_b, sp_b, dp_b);
      } else {
        // replicas differ modulo 16 (or many of them): one replica per pass
        for (int f = 0; f < nf; ++f) {
          uint8_t *one[1] = {pick<kGenFan>(dst, f)};
          copy_shifted_rows<1, RU>(src, one, 1, it.rows, run_b, sp_b, dp_b);
        }
      }
    }
#if RESHARD_GEN_SMEM_ITEM
    __syncthreads();  // everyone is done with s_item[buf]; s_item[buf ^ 1] is complete
#endif
  }
}

// Two builds of the general walker. reshard_copy_kernel (4 CTAs/SM) suits long single-row
// items; reshard_copy_rows_kernel (6 CTAs/SM, fewer registers) suits items of many short rows,
// where one warp walks one row and more resident warps hide more load latency.
// `wait_last`: the launch follows the aligned walker of the same pass, whose items touch other
// bytes; the grid then starts while that walker drains and takes its dependency wait just before
// it exits, so its completion still implies the aligned walker's (and the next launch on the
// stream, waiting for this grid, is ordered after both).
__global__ void __launch_bounds__(kBlock, RESHARD_GEN_MIN_BLOCKS) reshard_copy_kernel(
    const Item *__restrict__ items, const int32_t *__restrict__ idx, int n_items, const uint64_t *__restrict__ ptrs,
    const int32_t *__restrict__ gstart, const int32_t *__restrict__ mptr, const int64_t *__restrict__ moff,
    int wait_last) {
  if (!wait_last) pdl_enter();
  general_walk<kGenUnroll, RESHARD_GEN_ROW_UNROLL>(items, idx, n_items, ptrs, gstart, mptr, moff);
  if (wait_last) pdl_enter();
}

__global__ void __launch_bounds__(kBlock, RESHARD_ROWS_MIN_BLOCKS) reshard_copy_rows_kernel(
    const Item *__restrict__ items, const int32_t *__restrict__ idx, int n_items, const uint64_t *__restrict__ ptrs,
    const int32_t *__restrict__ gstart, const int32_t *__restrict__ mptr, const int64_t *__restrict__ moff,
    int wait_last) {
  if (!wait_last) pdl_enter();
  general_walk<RESHARD_ROWS_GEN_UNROLL, RESHARD_ROW_UNROLL>(items, idx, n_items, ptrs, gstart, mptr, moff);
  if (wait_last) pdl_enter();
}

// ------------------------------------------------------------------------ gather rows --

// One destination row assembled from two source pieces: row bytes [0, B) come from s0 (row byte
// b at s0 + b), bytes [B, rb) from s1 (row byte b at s1 + b - B). The row's destination words
// are taken piece by piece: piece 0's words (the first up to the one holding byte B - 1), then
// piece 1's (from the one holding byte B), so a word that holds the boundary is written twice,
// each time with only its own piece's bytes. Every word is one or two 16-byte block loads of its
// piece and a funnel shift by that piece's phase, as in copy_shifted_rows; the lanes of one row
// walk its words together. dst[f] are the row's starts in NF replicas with equal phase mod 16.
template <int NF, int RU>
__device__ __forceinline__ void gather_row(const uint8_t *s0, const uint8_t *s1, int B, int rb, uint8_t *const *dst,
                                           int nf, int lane) {
  const int a = (int)(reinterpret_cast<uintptr_t>(dst[0]) & 15);
  const int nw = (a + rb + 15) >> 4;   // destination words the row touches
  const int wb0 = (a + B - 1) >> 4;    // the last word with piece-0 bytes
  const int wb1 = (a + B) >> 4;        // the first word with piece-1 bytes
  const int nv = wb0 + 1 + nw - wb1;   // words of both pieces, the shared one twice
  const uintptr_t p0 = reinterpret_cast<uintptr_t>(s0) - a;      // source of word 0's byte 0, piece 0
  const uintptr_t p1 = reinterpret_cast<uintptr_t>(s1) - B - a;  // ... piece 1 (never read there)
  const int sh0 = (int)(p0 & 15), sh1 = (int)(p1 & 15);
  for (int v0 = lane; v0 < nv; v0 += 32 * RU) {
    uint4 lo[RU], hi[RU];
    int kmin[RU], kmax[RU], sh[RU], start[RU];
#pragma unroll
    for (int u = 0; u < RU; ++u) {
      const int v = v0 + 32 * u;
      kmin[u] = 16;
      kmax[u] = 0;
      sh[u] = 0;
      start[u] = 0;
      lo[u] = make_uint4(0, 0, 0, 0);
      hi[u] = make_uint4(0, 0, 0, 0);
      if (v < nv) {
        const bool second = v > wb0;
        const int w = second ? wb1 + (v - wb0 - 1) : v;
        const int st = 16 * w - a;  // row byte of the word's byte 0
        const int lo_b = second ? B : 0, hi_b = second ? rb : B;
        kmin[u] = max(lo_b - st, 0);
        kmax[u] = min(hi_b - st, 16);
        sh[u] = second ? sh1 : sh0;
        start[u] = st;
        const uint8_t *blk = reinterpret_cast<const uint8_t *>((second ? p1 : p0) - sh[u]) + 16 * w;
        if (kmin[u] < 16 - sh[u]) lo[u] = __ldg(reinterpret_cast<const uint4 *>(blk));
        if (sh[u] && kmax[u] > 16 - sh[u]) hi[u] = __ldg(reinterpret_cast<const uint4 *>(blk + 16));
      }
    }
#pragma unroll
    for (int u = 0; u < RU; ++u) {
      if (kmin[u] >= kmax[u]) continue;
      const uint4 o = sh[u] ? shift_bytes(lo[u], hi[u], sh[u]) : lo[u];
      if (kmin[u] == 0 && kmax[u] == 16) {
#pragma unroll
        for (int f = 0; f < NF; ++f)
          if (f < nf) store_stream(dst[f] + start[u], o);
      } else {
#pragma unroll
        for (int f = 0; f < NF; ++f)
          if (f < nf) store_partial(dst[f] + start[u], o, kmin[u], kmax[u]);
      }
    }
  }
}

#ifndef RESHARD_GATHER_UNROLL
#define RESHARD_GATHER_UNROLL RESHARD_ROW_UNROLL
#endif
#ifndef RESHARD_GATHER_MIN_BLOCKS
#define RESHARD_GATHER_MIN_BLOCKS RESHARD_ROWS_MIN_BLOCKS
#endif

// Gather items, resolved by the host for the current pointers: a persistent grid deals them
// round-robin (adjacent CTAs take adjacent items, so the grid streams through neighbouring rows)
// and each CTA's warps take an item's rows in turn. Descriptors are double-buffered in shared
// memory: 24 threads fetch the next one while the current one is copied. Replicas go two per
// pass when their phases agree mod 16, else one per pass. `wait_last` as in reshard_copy_kernel.
__global__ void __launch_bounds__(kBlock, RESHARD_GATHER_MIN_BLOCKS) reshard_copy_gather_kernel(
    const GBound *__restrict__ items, int n_items, const uint64_t *__restrict__ ptrs,
    const int32_t *__restrict__ gstart, const int32_t *__restrict__ mptr, const int64_t *__restrict__ moff,
    int wait_last) {
  if (!wait_last) pdl_enter();
  __shared__ GBound s_item[2];
  constexpr int kWords = (int)(sizeof(GBound) / sizeof(uint32_t));
  if (threadIdx.x < kWords && blockIdx.x < n_items)
    reinterpret_cast<uint32_t *>(&s_item[0])[threadIdx.x] =
        __ldg(reinterpret_cast<const uint32_t *>(items + blockIdx.x) + threadIdx.x);
  __syncthreads();
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  int buf = 0;
  for (int k = blockIdx.x; k < n_items; k += gridDim.x, buf ^= 1) {
    pdl_last_item(k, n_items);
    if (threadIdx.x < kWords && k + (int)gridDim.x < n_items)
      reinterpret_cast<uint32_t *>(&s_item[buf ^ 1])[threadIdx.x] =
          __ldg(reinterpret_cast<const uint32_t *>(items + k + gridDim.x) + threadIdx.x);
    const GBound &it = s_item[buf];
    const uint8_t *s0 = reinterpret_cast<const uint8_t *>(it.src[0]);
    const uint8_t *s1 = reinterpret_cast<const uint8_t *>(it.src[1]);
    const int B = it.B, rb = it.rb, rows = it.rows, nrep = it.nrep;
    const int64_t sp0 = it.sp[0], sp1 = it.sp[1], dp = it.dp[0];
    for (int f0 = 0; f0 < nrep; f0 += 2) {
      const int nf = min(2, nrep - f0);
      uint8_t *dst[2];
      if (f0 == 0) {
        dst[0] = reinterpret_cast<uint8_t *>(it.dst[0]);
        dst[1] = reinterpret_cast<uint8_t *>(it.dst[1]);
      } else {
        const int m = gstart[it.group] + f0;
        dst[0] = reinterpret_cast<uint8_t *>(ptrs[mptr[m]]) + moff[m] * it.esize + it.dst_off_b;
        dst[1] = nf > 1 ? reinterpret_cast<uint8_t *>(ptrs[mptr[m + 1]]) + moff[m + 1] * it.esize + it.dst_off_b : dst[0];
      }
      const bool same = ((reinterpret_cast<uintptr_t>(dst[0]) ^ reinterpret_cast<uintptr_t>(dst[1])) & 15) == 0;
      for (int r = warp; r < rows; r += kBlock / 32) {
        uint8_t *row[2] = {dst[0] + r * dp, dst[1] + r * dp};
        if (same) {
          gather_row<2, RESHARD_GATHER_UNROLL>(s0 + r * sp0, s1 + r * sp1, B, rb, row, nf, lane);
        } else {
          gather_row<1, RESHARD_GATHER_UNROLL>(s0 + r * sp0, s1 + r * sp1, B, rb, row, 1, lane);
          gather_row<1, RESHARD_GATHER_UNROLL>(s0 + r * sp0, s1 + r * sp1, B, rb, row + 1, 1, lane);
        }
      }
    }
    __syncthreads();  // everyone is done with s_item[buf]; s_item[buf ^ 1] is complete
  }
  if (wait_last) pdl_enter();
}

// One source row split into two destination rows (the pack pass's scatter items): row bytes
// [0, B) go to d0, bytes [B, rb) to d1, each destination on its own 16-byte word grid. The warp
// walks piece 0's destination words, then piece 1's; each word is one or two 16-byte block
// loads of the source row and a funnel shift by that piece's phase, as in gather_row.
template <int RU>
__device__ __forceinline__ void scatter_row(const uint8_t *s, int B, int rb, uint8_t *d0, uint8_t *d1, int lane) {
  const int a0 = (int)(reinterpret_cast<uintptr_t>(d0) & 15), a1 = (int)(reinterpret_cast<uintptr_t>(d1) & 15);
  const int len1 = rb - B;
  const int nw0 = (a0 + B + 15) >> 4;               // piece 0's destination words
  const int nv = nw0 + ((a1 + len1 + 15) >> 4);     // ... and piece 1's
  const uintptr_t p0 = reinterpret_cast<uintptr_t>(s) - a0;      // source of piece 0's word 0, byte 0
  const uintptr_t p1 = reinterpret_cast<uintptr_t>(s) + B - a1;  // ... piece 1's
  const int sh0 = (int)(p0 & 15), sh1 = (int)(p1 & 15);
  for (int v0 = lane; v0 < nv; v0 += 32 * RU) {
    uint4 lo[RU], hi[RU];
    int kmin[RU], kmax[RU], sh[RU], pos[RU];  // pos: 2 x (piece byte of the word's byte 0) + piece
#pragma unroll
    for (int u = 0; u < RU; ++u) {
      const int v = v0 + 32 * u;
      kmin[u] = 16;
      kmax[u] = 0;
      sh[u] = 0;
      pos[u] = 0;
      lo[u] = make_uint4(0, 0, 0, 0);
      hi[u] = make_uint4(0, 0, 0, 0);
      if (v < nv) {
        const bool second = v >= nw0;
        const int w = second ? v - nw0 : v;
        const int a = second ? a1 : a0, len = second ? len1 : B;
        const int st = 16 * w - a;  // piece byte of the word's byte 0
        kmin[u] = max(-st, 0);
        kmax[u] = min(len - st, 16);
        sh[u] = second ? sh1 : sh0;
        pos[u] = 2 * st + (second ? 1 : 0);
        const uint8_t *blk = reinterpret_cast<const uint8_t *>((second ? p1 : p0) - sh[u]) + 16 * w;
        if (kmin[u] < 16 - sh[u]) lo[u] = __ldg(reinterpret_cast<const uint4 *>(blk));
        if (sh[u] && kmax[u] > 16 - sh[u]) hi[u] = __ldg(reinterpret_cast<const uint4 *>(blk + 16));
      }
    }
#pragma unroll
    for (int u = 0; u < RU; ++u) {
      if (kmin[u] >= kmax[u]) continue;
      const uint4 o = sh[u] ? shift_bytes(lo[u], hi[u], sh[u]) : lo[u];
      uint8_t *dw = ((pos[u] & 1) ? d1 : d0) + (pos[u] >> 1);
      if (kmin[u] == 0 && kmax[u] == 16)
        store_stream(dw, o);
      else
        store_partial(dw, o, kmin[u], kmax[u]);
    }
  }
}

// Scatter items of the pack pass (one destination, the send buffer): dealt like the gather
// kernel's items, the rows of an item to the CTA's warps in turn.
// 4 CTAs/SM: the scatter walk fits 64 registers without spills (at 5 and 6 CTAs/SM it spills and
// measured 4-8% and 10-15% slower on the (2,4) mesh pack passes)
#ifndef RESHARD_SCATTER_MIN_BLOCKS
#define RESHARD_SCATTER_MIN_BLOCKS 4
#endif
__global__ void __launch_bounds__(kBlock, RESHARD_SCATTER_MIN_BLOCKS) reshard_copy_scatter_kernel(
    const GBound *__restrict__ items, int n_items, int wait_last) {
  if (!wait_last) pdl_enter();
  __shared__ GBound s_item[2];
  constexpr int kWords = (int)(sizeof(GBound) / sizeof(uint32_t));
  if (threadIdx.x < kWords && blockIdx.x < n_items)
    reinterpret_cast<uint32_t *>(&s_item[0])[threadIdx.x] =
        __ldg(reinterpret_cast<const uint32_t *>(items + blockIdx.x) + threadIdx.x);
  __syncthreads();
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  int buf = 0;
  for (int k = blockIdx.x; k < n_items; k += gridDim.x, buf ^= 1) {
    pdl_last_item(k, n_items);
    if (threadIdx.x < kWords && k + (int)gridDim.x < n_items)
      reinterpret_cast<uint32_t *>(&s_item[buf ^ 1])[threadIdx.x] =
          __ldg(reinterpret_cast<const uint32_t *>(items + k + gridDim.x) + threadIdx.x);
    const GBound &it = s_item[buf];
    const uint8_t *s = reinterpret_cast<const uint8_t *>(it.src[0]);
    uint8_t *d0 = reinterpret_cast<uint8_t *>(it.dst[0]);
    uint8_t *d1 = reinterpret_cast<uint8_t *>(it.dst[1]);
    const int B = it.B, rb = it.rb, rows = it.rows;
    const int64_t sp = it.sp[0], dp0 = it.dp[0], dp1 = it.dp[1];
    for (int r = warp; r < rows; r += kBlock / 32)
      scatter_row<RESHARD_GATHER_UNROLL>(s + r * sp, B, rb, d0 + r * dp0, d1 + r * dp1, lane);
    __syncthreads();  // everyone is done with s_item[buf]; s_item[buf ^ 1] is complete
  }
  if (wait_last) pdl_enter();
}

// The aligned walker: items the host found 16-byte aligned everywhere (sources, every replica,
// runs and pitches) for the current pointers; 16-byte copies only, more loads in flight. An
// item that is not aligned after all is skipped and reported in bit 1 of the status word.
__global__ void __launch_bounds__(kBlock, RESHARD_MIN_BLOCKS) reshard_copy_aligned_kernel(
    const Item *__restrict__ items, const int32_t *__restrict__ idx, int n_items, const uint64_t *__restrict__ ptrs,
    const int32_t *__restrict__ gstart, const int32_t *__restrict__ mptr, const int64_t *__restrict__ moff,
    int32_t *status) {
  pdl_enter();
  Item nxt;
  if (blockIdx.x < n_items) nxt = items[item_index(idx, blockIdx.x)];
  for (int k = blockIdx.x; k < n_items; k += gridDim.x) {
    pdl_last_item(k, n_items);
    const Item it = nxt;
    // the next item's descriptor is in flight while this one is copied
    if (k + (int)gridDim.x < n_items) nxt = items[item_index(idx, k + gridDim.x)];
    const int64_t es = it.esize;
    const uint8_t *src = reinterpret_cast<const uint8_t *>(ptrs[it.src]) + it.src_off * es;
    const int g0 = gstart[it.group];
    const int nrep = gstart[it.group + 1] - g0;
    const int64_t run_b = (int64_t)it.run * es;
    const int64_t sp_b = it.src_pitch * es, dp_b = it.dst_pitch * es;
    const uintptr_t geo = reinterpret_cast<uintptr_t>(src) | (uintptr_t)run_b |
                          (it.rows > 1 ? (uintptr_t)(sp_b | dp_b) : 0);
    for (int f0 = 0; f0 < nrep; f0 += kMaxFan) {
      const int nf = min(kMaxFan, nrep - f0);
      uint8_t *dst[kMaxFan];
      uintptr_t amask = geo;
#pragma unroll
      for (int f = 0; f < kMaxFan; ++f) {
        dst[f] = nullptr;
        if (f < nf) {
          const int m = g0 + f0 + f;
          dst[f] = reinterpret_cast<uint8_t *>(ptrs[mptr[m]]) + (moff[m] + it.dst_off) * es;
          amask |= reinterpret_cast<uintptr_t>(dst[f]);
        }
      }
      if ((amask & 15) == 0) {
        copy_aligned<kUnroll, kMaxFan>(src, dst, nf, it.rows, run_b, sp_b, dp_b);
      } else if (threadIdx.x == 0) {
        atomicOr(status, 2);
      }
    }
  }
}

// ------------------------------------------------- shared memory and bounded waits --

constexpr unsigned long long kWaitLimitNs = 200ull * 1000 * 1000;

__device__ __forceinline__ uint32_t smem_u32(const void *p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ unsigned long long global_ns() {
  unsigned long long t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

__device__ __forceinline__ bool bar_wait(uint32_t bar, uint32_t parity, unsigned long long deadline) {
  for (;;) {
    uint32_t ok;
    asm volatile(
        "{\n .reg .pred p;\n mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n selp.u32 %0, 1, 0, p;\n}"
        : "=r"(ok)
        : "r"(bar), "r"(parity)
        : "memory");
    if (ok) return true;
    if (global_ns() > deadline) return false;
  }
}

// ------------------------------------------------------- bulk-staged misaligned rows --
//
// reshard_copy_staged_kernel copies items of many short rows whose destination rows are not all
// 16-byte aligned (a column split whose row pitch is not a multiple of 16 bytes, for instance).
// Source rows are staged in shared memory by the TMA bulk-copy unit, and every warp runs its own
// pipeline, with no CTA-wide barrier: the rows of the CTA's items are dealt to its warps in
// chunks (as many rows as fit one stage); a warp issues one cp.async.bulk per row of a chunk
// (the row's span rounded out to 16-byte boundaries, so both ends stay in blocks that hold bytes
// of the row) into one of its stages, completion counted in bytes on that stage's mbarrier, and
// records in the stage's descriptor the row addresses it needs (source phase, every replica's
// destination row), so draining a stage reads no descriptor from global memory. Loads run up to
// kSStages - 1 chunks ahead and hold no registers while in flight. Draining: lane l writes
// destination words l, l + 32, ... of a row, each assembled from at most two aligned 16-byte
// shared-memory reads by a funnel shift, and stored whole (or, at the row's two ends, in
// naturally aligned pieces) to every replica. Waits are bounded like the transposing kernel's:
// on expiry bit 0 of the status word is set and the warp stops after waiting (bounded) for its
// copies in flight.

#ifndef RESHARD_STAGED
#define RESHARD_STAGED 1
#endif
#ifndef RESHARD_STAGED_STAGES
#define RESHARD_STAGED_STAGES 3
#endif
#ifndef RESHARD_STAGED_MAX_RUN
#define RESHARD_STAGED_MAX_RUN 4096
#endif
#ifndef RESHARD_STAGED_BYTES
#define RESHARD_STAGED_BYTES (RESHARD_STAGED_MAX_RUN + 64)
#endif
#ifndef RESHARD_STAGED_MIN_BLOCKS
#define RESHARD_STAGED_MIN_BLOCKS 2
#endif
constexpr int kSStages = RESHARD_STAGED_STAGES;   // stages per warp
constexpr int kSBytes = RESHARD_STAGED_BYTES;     // bytes per stage (multiple of 16)
constexpr int kSWarps = kBlock / 32;
constexpr size_t kStagedSmem = (size_t)kSWarps * kSStages * kSBytes;
static_assert(kSBytes % 16 == 0 && kSStages >= 2 && kSStages <= 8, "stage ring shape");
// rows up to this many bytes go through the staged kernel (one row and its rounding fit a stage)
constexpr int64_t kStagedMaxRun = RESHARD_STAGED_MAX_RUN;
static_assert(kStagedMaxRun + 32 <= kSBytes + 16, "a staged row and its rounding fit one stage");
constexpr int kStagedFan = kMaxFan;  // replicas an item may have to be staged
#ifndef RESHARD_STAGED_MIN_MB
#define RESHARD_STAGED_MIN_MB 512
#endif
// single-replica staged items run in the staged kernel only when they move at least this much
constexpr int64_t kStagedMinTraffic = (int64_t)RESHARD_STAGED_MIN_MB << 20;

struct StagedStage {
  uint64_t src;             // address of the chunk's first source row
  uint64_t dst[kStagedFan]; // every replica's destination row of the chunk's first row
  int64_t sp_b, dp_b;       // row pitches (bytes)
  int32_t run_b;            // bytes per row
  int32_t nrows;
  int32_t slot;             // bytes per row slot in the stage
  int32_t nrep;
};

__device__ __forceinline__ int staged_slot(int64_t run_b) { return (int)((run_b + 15) / 16 * 16 + 16); }

__device__ __forceinline__ uint4 lds16(const uint8_t *p) {
  uint4 v;
  asm volatile("ld.shared.v4.u32 {%0,%1,%2,%3}, [%4];" : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w) : "r"(smem_u32(p)));
  return v;
}

// Bytes [S, S + 16) of the 32-byte concatenation lo:hi, S a compile-time constant in [1, 16).
template <int S>
__device__ __forceinline__ uint4 shift_const(uint4 lo, uint4 hi) {
  const uint32_t v[8] = {lo.x, lo.y, lo.z, lo.w, hi.x, hi.y, hi.z, hi.w};
  constexpr int q = S / 4, r = (S % 4) * 8;
  uint4 o;
  if constexpr (r == 0) {
    o = make_uint4(v[q], v[q + 1], v[q + 2], v[q + 3]);
  } else {
    o.x = __funnelshift_r(v[q], v[q + 1], r);
    o.y = __funnelshift_r(v[q + 1], v[q + 2], r);
    o.z = __funnelshift_r(v[q + 2], v[q + 3], r);
    o.w = __funnelshift_r(v[q + 3], v[q + 4], r);
  }
  return o;
}

// Whole destination words [w0, w1) of a staged row at byte phase S: word w is bytes
// [16 w + S, 16 w + S + 16) of the stage from sw0 (one aligned read when S == 0, two otherwise).
#ifndef RESHARD_STAGED_UNROLL
#define RESHARD_STAGED_UNROLL 4
#endif
template <int S, int NF>
__device__ __forceinline__ void drain_words(const uint8_t *sw0, uint8_t *d0, uint8_t *d1, int w0, int w1, int lane) {
  constexpr int U = RESHARD_STAGED_UNROLL;  // words per lane whose shared reads are in flight together
  for (int w = w0 + lane; w < w1; w += 32 * U) {
    uint4 lo[U], hi[U];
#pragma unroll
    for (int u = 0; u < U; ++u) {
      const int x = w + 32 * u;
      lo[u] = make_uint4(0, 0, 0, 0);
      hi[u] = make_uint4(0, 0, 0, 0);
      if (x < w1) {
        lo[u] = lds16(sw0 + 16 * x);
        if constexpr (S != 0) hi[u] = lds16(sw0 + 16 * x + 16);
      }
    }
#pragma unroll
    for (int u = 0; u < U; ++u) {
      const int x = w + 32 * u;
      if (x < w1) {
        uint4 o;
        if constexpr (S == 0)
          o = lo[u];
        else
          o = shift_const<S>(lo[u], hi[u]);
        store_stream(d0 + 16 * x, o);
        if constexpr (NF == 2) store_stream(d1 + 16 * x, o);
      }
    }
  }
}

// Whole words of a row to one destination (d1 == nullptr) or to two at the same byte phase.
__device__ __forceinline__ void drain_words_at(int s, const uint8_t *sw0, uint8_t *d0, uint8_t *d1, int w0, int w1,
                                               int lane) {
#define RESHARD_DRAIN_CASE(S_)                                       \
  case S_:                                                           \
    if (d1)                                                          \
      drain_words<S_, 2>(sw0, d0, d1, w0, w1, lane);                 \
    else                                                             \
      drain_words<S_, 1>(sw0, d0, nullptr, w0, w1, lane);            \
    break;
  switch (s) {
    RESHARD_DRAIN_CASE(0) RESHARD_DRAIN_CASE(1) RESHARD_DRAIN_CASE(2) RESHARD_DRAIN_CASE(3)
    RESHARD_DRAIN_CASE(4) RESHARD_DRAIN_CASE(5) RESHARD_DRAIN_CASE(6) RESHARD_DRAIN_CASE(7)
    RESHARD_DRAIN_CASE(8) RESHARD_DRAIN_CASE(9) RESHARD_DRAIN_CASE(10) RESHARD_DRAIN_CASE(11)
    RESHARD_DRAIN_CASE(12) RESHARD_DRAIN_CASE(13) RESHARD_DRAIN_CASE(14) default:
    RESHARD_DRAIN_CASE(15)
  }
#undef RESHARD_DRAIN_CASE
}

__global__ void __launch_bounds__(kBlock, RESHARD_STAGED_MIN_BLOCKS) reshard_copy_staged_kernel(
    const Item *__restrict__ items, const int32_t *__restrict__ idx, int n_items, const uint64_t *__restrict__ ptrs,
    const int32_t *__restrict__ gstart, const int32_t *__restrict__ mptr, const int64_t *__restrict__ moff,
    int32_t *status, int wait_last) {
  if (!wait_last) pdl_enter();
  extern __shared__ __align__(128) uint8_t sring[];
  __shared__ __align__(8) uint64_t bar[kSWarps][kSStages];
  __shared__ StagedStage desc[kSWarps][kSStages];
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  uint8_t *ring = sring + (size_t)warp * kSStages * kSBytes;
  if (lane == 0) {
    for (int st = 0; st < kSStages; ++st) asm volatile("mbarrier.init.shared::cta.b64 [%0], 1;" ::"r"(smem_u32(&bar[warp][st])));
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  __syncwarp();

  // issue cursor of this warp: item k (position in the launch's list), chunk j of that item;
  // chunks of rows are dealt to the warps in turn, chunk j to warp j % kSWarps
  int ik = blockIdx.x, ij = warp;
  Item it{};
  int rpc = 1, nch = 0;  // rows per chunk and chunks of the current item
  auto load_item = [&]() {
    while (ik < n_items) {
      it = items[item_index(idx, ik)];
      rpc = kSBytes / staged_slot((int64_t)it.run * it.esize);
      nch = (it.rows + rpc - 1) / rpc;
      if (ij < nch) return;
      ij -= nch;  // keep the deal going across items: chunk numbering continues
      ik += gridDim.x;
    }
  };
  load_item();
  auto issue = [&](int st) -> bool {
    if (ik >= n_items) return false;
    const int64_t es = it.esize, run_b = (int64_t)it.run * es, sp_b = it.src_pitch * es;
    const int slot = staged_slot(run_b);
    const int r0 = ij * rpc, n = min(rpc, it.rows - r0);
    const uintptr_t src0 = (uintptr_t)ptrs[it.src] + (uintptr_t)((it.src_off + (int64_t)r0 * it.src_pitch) * es);
    const int g0 = gstart[it.group], nrep = gstart[it.group + 1] - g0;
    StagedStage &d = desc[warp][st];
    if (lane < nrep)
      d.dst[lane] = (uint64_t)ptrs[mptr[g0 + lane]] + (uint64_t)((moff[g0 + lane] + it.dst_off + (int64_t)r0 * it.dst_pitch) * es);
    uint32_t tx = 0;
    for (int r = lane; r < n; r += 32) {
      const uintptr_t a = src0 + (uintptr_t)(r * sp_b);
      tx += (uint32_t)(((a + run_b + 15) & ~(uintptr_t)15) - (a & ~(uintptr_t)15));
    }
    tx = __reduce_add_sync(0xffffffffu, tx);
    const uint32_t b = smem_u32(&bar[warp][st]);
    if (lane == 0) {
      d.src = src0;
      d.sp_b = sp_b;
      d.dp_b = it.dst_pitch * es;
      d.run_b = (int32_t)run_b;
      d.nrows = n;
      d.slot = slot;
      d.nrep = nrep;
      asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(b), "r"(tx) : "memory");
    }
    __syncwarp();
    uint8_t *dst0 = ring + (size_t)st * kSBytes;
    for (int r = lane; r < n; r += 32) {
      const uintptr_t a = src0 + (uintptr_t)(r * sp_b);
      const uintptr_t lo = a & ~(uintptr_t)15, hi = (a + run_b + 15) & ~(uintptr_t)15;
      asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
                       smem_u32(dst0 + (size_t)r * slot)),
                   "l"(lo), "r"((uint32_t)(hi - lo)), "r"(b)
                   : "memory");
    }
    // next chunk of this warp
    ij += kSWarps;
    if (ij >= nch) {
      ij -= nch;
      ik += gridDim.x;
      load_item();
    }
    return true;
  };

  int issued = 0;
  for (int st = 0; st < kSStages; ++st)
    if (issue(st)) ++issued;
  uint32_t phases = 0;
  for (int t = 0; t < issued; ++t) {
    const int st = t % kSStages;
#if RESHARD_PDL
    if (t + 1 == issued && ik >= n_items) asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
#endif
    if (!bar_wait(smem_u32(&bar[warp][st]), (phases >> st) & 1, global_ns() + kWaitLimitNs)) {
      // a bulk load never completed: report, give this warp's loads in flight one more bounded
      // wait, and stop (the launch's output is incomplete)
      if (lane == 0) atomicOr(status, 1);
      for (int u = t; u < issued; ++u) {
        const int su = u % kSStages;
        bar_wait(smem_u32(&bar[warp][su]), (phases >> su) & 1, global_ns() + kWaitLimitNs);
      }
      break;
    }
    phases ^= 1u << st;
    const StagedStage &d = desc[warp][st];
    const uintptr_t src0 = (uintptr_t)d.src;
    const int64_t sp_b = d.sp_b, dp_b = d.dp_b;
    const int run_b = d.run_b, nrows = d.nrows, slot = d.slot, nrep = d.nrep;
    const uint8_t *stg = ring + (size_t)st * kSBytes;
    for (int r = 0; r < nrows; ++r) {
      const uint8_t *srow = stg + (size_t)r * slot;                   // the row from its 16-byte block
      const int sh0 = (int)((src0 + (uintptr_t)(r * sp_b)) & 15);     // row byte 0 sits at srow + sh0
      for (int f = 0; f < nrep; ++f) {
        uint8_t *drow = reinterpret_cast<uint8_t *>(d.dst[f]) + r * dp_b;
        const int a = (int)(reinterpret_cast<uintptr_t>(drow) & 15);
        const int nw = (a + run_b + 15) >> 4;
        const int s = (sh0 - a) & 15;  // byte phase of every destination word in the stage
        uint8_t *dword0 = drow - a;
        const uint8_t *sw0 = srow + (sh0 - a - s);  // stage bytes of word 0 start here (or 16 before srow)
        // whole words [wf, wl): the first word is whole when the row starts aligned, the last
        // when the row ends on a word boundary; the next replica's words too when it has the same
        // byte phase (each word is then read and shifted once for both)
        const int wf = a ? 1 : 0, wl = (a + run_b) >> 4;
        uint8_t *pair = nullptr;
        if (f + 1 < nrep) {
          uint8_t *drow1 = reinterpret_cast<uint8_t *>(d.dst[f + 1]) + r * dp_b;
          if ((reinterpret_cast<uintptr_t>(drow1) & 15) == (uintptr_t)a) pair = drow1 - a;
        }
        if (wl > wf) drain_words_at(s, sw0, dword0, pair, wf, wl, lane);
        // the row's first and last word when partial (one lane each): only bytes [kmin, kmax)
        // belong to the row, and only aligned stage blocks that hold some of them are read
        int w = -1;
        if (lane == 0 && a) w = 0;
        if (lane == 1 && wl < nw && (wl > 0 || !a)) w = wl;
        if (w >= 0) {
          const int start = 16 * w - a;
          const int kmin = w == 0 ? a : 0;
          const int kmax = run_b - start < 16 ? run_b - start : 16;
          uint4 lo = make_uint4(0, 0, 0, 0), hi = make_uint4(0, 0, 0, 0);
          if (kmin < 16 - s) lo = lds16(sw0 + 16 * w);
          if (s && kmax > 16 - s) hi = lds16(sw0 + 16 * w + 16);
          const uint4 o = s ? shift_bytes(lo, hi, s) : lo;
          store_partial(dword0 + 16 * w, o, kmin, kmax);
          if (pair) store_partial(pair + 16 * w, o, kmin, kmax);
        }
        if (pair) ++f;  // that replica is written too
      }
    }
    __syncwarp();  // the stage is drained: refill it
    if (issue(st)) ++issued;
  }
  if (wait_last) pdl_enter();
}

// ------------------------------------------------------------------------ MXFP8 epilogue --

// Shared E8M0 exponent X of a block from its largest BF16 magnitude (15-bit pattern, finite):
// X = floor(log2 amax) - 8, clamped to [-127, 127]; an all-zero block takes -127.
__device__ __forceinline__ int block_exponent(uint32_t amax) {
  if (amax == 0) return -127;
  const int e = (int)(amax >> 7);
  const int lg = e ? e - 127 : -133 + (31 - __clz((int)amax));
  return max(-127, min(127, lg - 8));
}

// Two floats -> two E4M3 bytes (RNE, saturating to +-448); `lo` lands in the low byte.
__device__ __forceinline__ uint32_t cvt_e4m3x2(float lo, float hi) {
  unsigned short r;
  asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(r) : "f"(hi), "f"(lo));
  return (uint32_t)r;
}

__device__ __forceinline__ float bf16_lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t w) { return __uint_as_float(w & 0xFFFF0000u); }


#ifndef RESHARD_MXFP8_UNROLL
#define RESHARD_MXFP8_UNROLL 2
#endif
#ifndef RESHARD_MXFP8_MIN_BLOCKS
#define RESHARD_MXFP8_MIN_BLOCKS 4
#endif
#ifndef RESHARD_MXFP8_BLOCK
#define RESHARD_MXFP8_BLOCK 256
#endif
#ifndef RESHARD_MXFP8_ELEMS
#define RESHARD_MXFP8_ELEMS 16
#endif
#ifndef RESHARD_MXFP8_FAN
#define RESHARD_MXFP8_FAN 2
#endif
#ifndef RESHARD_MXFP8_WIDE
#define RESHARD_MXFP8_WIDE 1
#endif
constexpr int kQBlock = RESHARD_MXFP8_BLOCK;    // threads per CTA
constexpr int kQUnroll = RESHARD_MXFP8_UNROLL;  // lane slots in flight per thread
constexpr int kQE = RESHARD_MXFP8_ELEMS;        // BF16 elements per lane slot (8 or 16)
constexpr int kQV = kQE / 8;                    // 16-byte loads per slot
constexpr int kQLanes = 32 / kQE;               // lanes sharing one 32-element block
constexpr int kQMaxFan = RESHARD_MXFP8_FAN;      // replicas per pass (pointer pairs in registers)
static_assert(kQE == 8 || kQE == 16, "a lane holds 8 or 16 elements of a 32-element block");

// Per-halfword unsigned max of two packed 16-bit pairs.
__device__ __forceinline__ uint32_t max_u16x2(uint32_t a, uint32_t b) {
  uint32_t r;
  asm("max.u16x2 %0, %1, %2;" : "=r"(r) : "r"(a), "r"(b));
  return r;
}

// Largest BF16 magnitude (15-bit pattern) among the 8 values of a 16-byte load, folded into
// the running packed maximum `m` (two halfword lanes, combined by amax_of).
__device__ __forceinline__ uint32_t fold_mag8(uint32_t m, uint4 v) {
  m = max_u16x2(m, v.x & 0x7FFF7FFFu);
  m = max_u16x2(m, v.y & 0x7FFF7FFFu);
  m = max_u16x2(m, v.z & 0x7FFF7FFFu);
  return max_u16x2(m, v.w & 0x7FFF7FFFu);
}

__device__ __forceinline__ uint32_t amax_of(uint32_t m) { return max(m & 0xFFFFu, m >> 16); }

// Quantize 8 BF16 values (one 16-byte load) by 2^-X, `inv` = 2^-X of the block.
__device__ __forceinline__ uint2 quantize8_by(uint4 v, float inv) {
  uint2 q;
  q.x = cvt_e4m3x2(bf16_lo(v.x) * inv, bf16_hi(v.x) * inv) | (cvt_e4m3x2(bf16_lo(v.y) * inv, bf16_hi(v.y) * inv) << 16);
  q.y = cvt_e4m3x2(bf16_lo(v.z) * inv, bf16_hi(v.z) * inv) | (cvt_e4m3x2(bf16_lo(v.w) * inv, bf16_hi(v.w) * inv) << 16);
  return q;
}

__device__ __forceinline__ uint4 load_bf16x8(const uint8_t *p, bool vec) {
  if (vec) return load_stream(p);
  const uint16_t *h = reinterpret_cast<const uint16_t *>(p);
  return make_uint4((uint32_t)h[0] | ((uint32_t)h[1] << 16), (uint32_t)h[2] | ((uint32_t)h[3] << 16),
                    (uint32_t)h[4] | ((uint32_t)h[5] << 16), (uint32_t)h[6] | ((uint32_t)h[7] << 16));
}

__device__ __forceinline__ void store_bytes(uint8_t *p, uint32_t w) {
#pragma unroll
  for (int k = 0; k < 4; ++k) p[k] = (uint8_t)(w >> (8 * k));
}

__global__ void __launch_bounds__(kQBlock, RESHARD_MXFP8_MIN_BLOCKS) reshard_mxfp8_kernel(
    const Item *__restrict__ items, int n_items, const uint64_t *__restrict__ ptrs, const int32_t *__restrict__ gstart,
    const int32_t *__restrict__ mptr, const int64_t *__restrict__ moff, int64_t n_dst_ptrs) {
  pdl_enter();
  const int lane = threadIdx.x & 31;
  for (int i = blockIdx.x; i < n_items; i += gridDim.x) {
    pdl_last_item(i, n_items);
    const Item it = items[i];
    const uint8_t *src = reinterpret_cast<const uint8_t *>(ptrs[it.src]) + it.src_off * 2;
    const int g0 = gstart[it.group];
    const int nrep = gstart[it.group + 1] - g0;
    const int per_row = it.run / kQE;  // lane slots per row; a multiple of kQLanes
    const int total = it.rows * per_row;
    const int64_t sp_b = it.src_pitch * 2;
    const bool vec = ((reinterpret_cast<uintptr_t>(src) | (it.rows > 1 ? (uintptr_t)sp_b : 0)) & 15) == 0;
    const bool vec32 = ((reinterpret_cast<uintptr_t>(src) | (it.rows > 1 ? (uintptr_t)sp_b : 0)) & 31) == 0;
    for (int f0 = 0; f0 < nrep; f0 += kQMaxFan) {
      const int nf = min(kQMaxFan, nrep - f0);
      uint8_t *dq[kQMaxFan];
      uint8_t *ds[kQMaxFan];
      uintptr_t amask = it.rows > 1 ? (uintptr_t)it.dst_pitch : 0;
#pragma unroll
      for (int f = 0; f < kQMaxFan; ++f) {
        dq[f] = nullptr;
        ds[f] = nullptr;
        if (f < nf) {
          const int m = g0 + f0 + f;
          const int64_t e0 = moff[m] + it.dst_off;  // element offset of the item in the shard buffer
          dq[f] = reinterpret_cast<uint8_t *>(ptrs[mptr[m]]) + e0;
          ds[f] = reinterpret_cast<uint8_t *>(ptrs[mptr[m] + n_dst_ptrs]) + e0 / 32;
          amask |= reinterpret_cast<uintptr_t>(dq[f]);
        }
      }
      const bool stv = (amask & (kQE - 1)) == 0;  // one kQE-byte store per slot
      // slot j of the item is (row j / per_row, lane slot j % per_row); each pass advances every
      // slot of this thread by kStride, so (row, slot) step by a quotient and remainder taken
      // once per item instead of a division per slot
      constexpr int kStride = kQBlock * kQUnroll;
      const int q_step = kStride / per_row, r_step = kStride - q_step * per_row;
      const int q_blk = kQBlock / per_row, r_blk = kQBlock - q_blk * per_row;  // slot u + 1 from slot u
      int row0 = (int)threadIdx.x / per_row;
      int col0 = (int)threadIdx.x - row0 * per_row;
      // j0 is warp-uniform, so every lane takes part in every shuffle
      for (int j0 = threadIdx.x - lane; j0 < total; j0 += kStride) {
        uint4 v[kQUnroll][kQV];
        int64_t eoff[kQUnroll];  // element offset of this slot's first value within the item
#pragma unroll
        for (int u = 0; u < kQUnroll; ++u) {
          const int j = j0 + u * kQBlock + lane;
#pragma unroll
          for (int k = 0; k < kQV; ++k) v[u][k] = make_uint4(0, 0, 0, 0);
          eoff[u] = -1;
          int r = row0, o = col0;
#pragma unroll
          for (int w = 0; w < u; ++w) {
            o += r_blk;
            r += q_blk;
            if (o >= per_row) {
              o -= per_row;
              ++r;
            }
          }
          if (j < total) {
            const uint8_t *p = src + r * sp_b + 2 * kQE * (int64_t)o;
            eoff[u] = r * it.dst_pitch + kQE * (int64_t)o;
            if (RESHARD_MXFP8_WIDE && kQV == 2 && vec32) {
              load_stream32(p, v[u][0], v[u][kQV - 1]);
            } else {
#pragma unroll
              for (int k = 0; k < kQV; ++k) v[u][k] = load_bf16x8(p + 16 * k, vec);
            }
          }
        }
        col0 += r_step;
        row0 += q_step;
        if (col0 >= per_row) {
          col0 -= per_row;
          ++row0;
        }
#pragma unroll
        for (int u = 0; u < kQUnroll; ++u) {
          uint32_t m = 0;
#pragma unroll
          for (int k = 0; k < kQV; ++k) m = fold_mag8(m, v[u][k]);
          uint32_t amax = amax_of(m);
#pragma unroll
          for (int s = 1; s < kQLanes; s <<= 1) amax = max(amax, __shfl_xor_sync(0xffffffffu, amax, s));
          if (eoff[u] < 0) continue;
          uint2 q[kQV];
          const bool special = amax >= 0x7F80u;  // Inf/NaN in the block: E4M3 NaN, scale NaN
          const int x = block_exponent(amax);
          const float inv = __uint_as_float((uint32_t)(127 - x) << 23);  // 2^-X, X in [-127, 119]
#pragma unroll
          for (int k = 0; k < kQV; ++k)
            q[k] = special ? make_uint2(0x7F7F7F7Fu, 0x7F7F7F7Fu) : quantize8_by(v[u][k], inv);
          const uint32_t sbyte = special ? 0xFFu : (uint32_t)(x + 127);
#pragma unroll
          for (int f = 0; f < kQMaxFan; ++f) {
            if (f < nf) {
              uint8_t *p = dq[f] + eoff[u];
              if (stv) {
                if constexpr (kQV == 2)
                  __stcs(reinterpret_cast<uint4 *>(p), make_uint4(q[0].x, q[0].y, q[kQV - 1].x, q[kQV - 1].y));
                else
                  __stcs(reinterpret_cast<uint2 *>(p), q[0]);
              } else {
#pragma unroll
                for (int k = 0; k < kQV; ++k) {
                  store_bytes(p + 8 * k, q[k].x);
                  store_bytes(p + 8 * k + 4, q[k].y);
                }
              }
              if ((lane & (kQLanes - 1)) == 0) ds[f][eoff[u] / 32] = (uint8_t)sbyte;
            }
          }
        }
      }
    }
  }
}

// ----------------------------------------------------------- transposing copy (TMA) --
//
// reshard_transpose_kernel moves regions whose source is contiguous along one dim (C) and whose
// destination is contiguous along another (R): a transposed layout on one side. Tiles of
// 128 rows (R) x 128 bytes (C) are staged in shared memory by TMA 2-D box loads
// (cp.async.bulk.tensor, 128-byte swizzle, mbarrier completion, two stages in flight); each
// thread then reads 32 bytes' worth of one column down the tile (conflict-free thanks to the
// swizzle) and stores them as one contiguous 32-byte run of the destination. Where a slab's
// tensor map could not be encoded (base or pitch not 16-byte aligned), the tile is filled by
// plain loads instead. Every wait on an mbarrier is bounded; on timeout the kernel sets bit 0
// of the plan's status word and returns.

constexpr int kTBlock = 256;                          // threads per CTA (one unit per tile per thread)
constexpr int kTStages = 2;
constexpr int kTileBytes = kTileRows * kTileRowBytes;  // 16 KiB per stage
// Byte offset in a 128-byte-swizzled tile of (row, byte within the row).
__device__ __forceinline__ int swz(int row, int byte) { return row * kTileRowBytes + ((((byte >> 4) ^ (row & 7))) << 4) + (byte & 15); }

// Fill one tile with plain loads (same swizzled layout as TMA). Column x of the tile is slab
// column x0 + x; only elements inside the item are read, the rest become zero.
template <int ES>
__device__ __forceinline__ void tile_fill_plain(uint8_t *tile, const TItem &it, const uint8_t *src, int x0, int y0) {
  constexpr int TC = kTileRowBytes / ES;
  for (int e = threadIdx.x; e < kTileRows * TC; e += kTBlock) {
    const int row = e / TC, col = e - row * TC;
    const int xs = x0 + col - it.x, ys = y0 + row - it.y;  // item-relative
    uint8_t v[ES];
#pragma unroll
    for (int b = 0; b < ES; ++b) v[b] = 0;
    if (xs >= 0 && xs < it.cols && ys >= 0 && ys < it.rows) {
      const uint8_t *g = src + ((int64_t)ys * it.src_pitch + xs) * ES;
#pragma unroll
      for (int b = 0; b < ES; ++b) v[b] = g[b];
    }
    uint8_t *d = tile + swz(row, col * ES);
#pragma unroll
    for (int b = 0; b < ES; ++b) d[b] = v[b];
  }
}

__device__ __forceinline__ void store32(uint8_t *p, const uint32_t *w) {
  asm volatile("st.global.cs.v8.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8};" ::"l"(p), "r"(w[0]), "r"(w[1]), "r"(w[2]),
               "r"(w[3]), "r"(w[4]), "r"(w[5]), "r"(w[6]), "r"(w[7])
               : "memory");
}

// One tile to the destinations. A thread owns CPT adjacent columns (one 4-byte shared word per
// row; 8 bytes for 8-byte elements) and RPC rows: 32 bytes of each column, which it writes as
// one contiguous 32-byte run of the destination (one 256-bit store when aligned). Lanes of a warp
// take consecutive column groups of one row chunk: with the 128-byte swizzle their shared reads
// hit 32 different banks.
template <int ES>
__device__ __forceinline__ void tile_store(const uint8_t *tile, const TItem &it, uint8_t *const *dst, int nf, int x0,
                                           int y0) {
  constexpr int TC = kTileRowBytes / ES;          // columns per tile
  constexpr int CPT = ES >= 4 ? 1 : 4 / ES;       // columns per thread
  constexpr int RPC = 32 / ES;                    // rows per thread (32 bytes per column)
  constexpr int NG = TC / CPT;                    // column groups per tile
  constexpr int UNITS = NG * (kTileRows / RPC);
  for (int u = threadIdx.x; u < UNITS; u += kTBlock) {
    const int g = u % NG, chunk = u / NG;
    const int r0 = y0 + chunk * RPC - it.y;       // item row of the first element
    const int c0 = x0 + g * CPT - it.x;           // item column of the first column
    if (r0 >= it.rows || c0 + CPT <= 0 || c0 >= it.cols) continue;
    uint32_t w[CPT][8];
#pragma unroll
    for (int k = 0; k < RPC; ++k) {
      const int row = chunk * RPC + k;
      if constexpr (ES == 8) {
        const uint2 v = *reinterpret_cast<const uint2 *>(tile + swz(row, g * 8));
        w[0][2 * k] = v.x;
        w[0][2 * k + 1] = v.y;
      } else {
        const uint32_t v = *reinterpret_cast<const uint32_t *>(tile + swz(row, g * 4));
#pragma unroll
        for (int j = 0; j < CPT; ++j) {
          if constexpr (ES == 4) {
            w[j][k] = v;
          } else if constexpr (ES == 2) {
            const uint32_t h = (v >> (16 * j)) & 0xFFFFu;
            w[j][k / 2] = (k & 1) ? (w[j][k / 2] | (h << 16)) : h;
          } else {
            const uint32_t b = (v >> (8 * j)) & 0xFFu;
            w[j][k / 4] = (k & 3) ? (w[j][k / 4] | (b << (8 * (k & 3)))) : b;
          }
        }
      }
    }
    const int nvalid = min(RPC, it.rows - r0);
#pragma unroll
    for (int j = 0; j < CPT; ++j) {
      const int c = c0 + j;
      if (c < 0 || c >= it.cols) continue;
      const int64_t eoff = it.dst_off + (int64_t)c * it.dst_pitch + r0;
#pragma unroll
      for (int f = 0; f < kMaxFan; ++f) {
        if (f >= nf) break;
        uint8_t *p = dst[f] + eoff * ES;
        const uintptr_t a = reinterpret_cast<uintptr_t>(p);
        if (nvalid == RPC && (a & 31) == 0) {
          store32(p, w[j]);
        } else if (nvalid == RPC && (a & 15) == 0) {
          store_stream(p, make_uint4(w[j][0], w[j][1], w[j][2], w[j][3]));
          store_stream(p + 16, make_uint4(w[j][4], w[j][5], w[j][6], w[j][7]));
        } else {
          const int nb = nvalid * ES;
#pragma unroll
          for (int q = 0; q < 8; ++q)
#pragma unroll
            for (int bb = 0; bb < 4; ++bb)
              if (4 * q + bb < nb) p[4 * q + bb] = (uint8_t)(w[j][q] >> (8 * bb));
        }
      }
    }
  }
}

template <int ES>
__device__ void transpose_item(const TItem &it, const uint8_t *src, uint8_t *const *dst, int nf, const CUtensorMap *map,
                               bool tma, uint8_t (*tile)[kTileBytes], uint64_t *bar, uint32_t &phases,
                               int32_t *status, bool &abort) {
  constexpr int TC = kTileRowBytes / ES;
  constexpr int XAL = 16 / ES;                 // TMA box x must start on a 16-byte boundary
  const int xa = it.x / XAL * XAL;             // first tile's slab column
  const int ntc = (it.x + it.cols - xa + TC - 1) / TC;
  const int ntr = (it.rows + kTileRows - 1) / kTileRows;
  const int nt = ntc * ntr;
  if (!tma) {
    for (int t = 0; t < nt; ++t) {
      const int x0 = xa + (t % ntc) * TC, y0 = it.y + (t / ntc) * kTileRows;
      __syncthreads();
      tile_fill_plain<ES>(tile[0], it, src, x0, y0);
      __syncthreads();
      tile_store<ES>(tile[0], it, dst, nf, x0, y0);
    }
    __syncthreads();
    return;
  }
  auto issue = [&](int t, int stage) {
    if (threadIdx.x == 0) {
      const int x0 = xa + (t % ntc) * TC, y0 = it.y + (t / ntc) * kTileRows;
      const uint32_t b = smem_u32(&bar[stage]);
      asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(b), "r"(kTileBytes) : "memory");
      asm volatile(
          "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3}], [%4];" ::"r"(
              smem_u32(tile[stage])),
          "l"(reinterpret_cast<uint64_t>(map)), "r"(x0), "r"(y0), "r"(b)
          : "memory");
    }
  };
  if (threadIdx.x == 0)
    asm volatile("fence.proxy.tensormap::generic.acquire.gpu [%0], 128;" ::"l"(reinterpret_cast<uint64_t>(map)) : "memory");
  issue(0, 0);
  for (int t = 0; t < nt; ++t) {
    const int stage = t & 1;
    if (t + 1 < nt) issue(t + 1, stage ^ 1);
    const uint32_t parity = (phases >> stage) & 1;
    const bool ok = bar_wait(smem_u32(&bar[stage]), parity, global_ns() + kWaitLimitNs);
    if (__syncthreads_or(!ok)) {
      // a TMA load never completed: report, give the copies in flight one more bounded wait, stop
      if (threadIdx.x == 0) atomicOr(status, 1);
      bar_wait(smem_u32(&bar[stage]), parity, global_ns() + kWaitLimitNs);
      if (t + 1 < nt) bar_wait(smem_u32(&bar[stage ^ 1]), (phases >> (stage ^ 1)) & 1, global_ns() + kWaitLimitNs);
      abort = true;
      return;
    }
    phases ^= 1u << stage;
    const int x0 = xa + (t % ntc) * TC, y0 = it.y + (t / ntc) * kTileRows;
    tile_store<ES>(tile[stage], it, dst, nf, x0, y0);
    __syncthreads();  // the stage is free for the load two tiles ahead
  }
}

// One build per element size ES (the planner groups transposing items by element size and the
// host launches each group with its build): a single-size kernel keeps its register assembly in
// registers and measured 1.6% faster than one that switches on the size per item.
template <int ES>
__global__ void __launch_bounds__(kTBlock, 2) reshard_transpose_kernel(
    const TItem *__restrict__ items, int n_items, const uint64_t *__restrict__ ptrs, const int32_t *__restrict__ gstart,
    const int32_t *__restrict__ mptr, const int64_t *__restrict__ moff, const CUtensorMap *__restrict__ maps,
    const int32_t *__restrict__ map_ok, int32_t *status) {
  pdl_enter();
  __shared__ __align__(1024) uint8_t tile[kTStages][kTileBytes];
  __shared__ __align__(8) uint64_t bar[kTStages];
  if (threadIdx.x == 0) {
    for (int s = 0; s < kTStages; ++s) asm volatile("mbarrier.init.shared::cta.b64 [%0], 1;" ::"r"(smem_u32(&bar[s])));
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  __syncthreads();
  uint32_t phases = 0;  // expected parity bit per stage
  bool abort = false;
  for (int i = blockIdx.x; i < n_items && !abort; i += gridDim.x) {
    pdl_last_item(i, n_items);
    const TItem it = items[i];
    const uint8_t *src = reinterpret_cast<const uint8_t *>(ptrs[it.src]) + it.src_off * it.esize;
    const bool tma = it.map >= 0 && map_ok[it.map];
    const CUtensorMap *map = tma ? maps + it.map : nullptr;
    const int g0 = gstart[it.group];
    const int nrep = gstart[it.group + 1] - g0;
    for (int f0 = 0; f0 < nrep && !abort; f0 += kMaxFan) {
      const int nf = min(kMaxFan, nrep - f0);
      uint8_t *dst[kMaxFan];
#pragma unroll
      for (int f = 0; f < kMaxFan; ++f) {
        dst[f] = nullptr;
        if (f < nf) dst[f] = reinterpret_cast<uint8_t *>(ptrs[mptr[g0 + f0 + f]]) + moff[g0 + f0 + f] * it.esize;
      }
      transpose_item<ES>(it, src, dst, nf, map, tma, tile, bar, phases, status, abort);
    }
  }
}

// -------------------------------------------------------------- bulk copy walker (TMA) --
//
// reshard_bulk_kernel copies aligned items with the TMA bulk-copy unit instead of load/store
// instructions: one thread per CTA walks its items as (row, chunk) pieces of up to kBulkChunk
// bytes, loads each piece into a ring of shared-memory stages (cp.async.bulk, completion on an
// mbarrier), and writes it to every replica with bulk stores (one bulk group per piece). Loads
// run kBulkStages - 1 pieces ahead; a stage is reloaded only after the stores that read it are
// done reading (cp.async.bulk.wait_group.read). Waits on the mbarriers are bounded like the
// transposing kernel's (status bit 0).

#ifndef RESHARD_BULK
#define RESHARD_BULK 0
#endif
#ifndef RESHARD_BULK_STAGES
#define RESHARD_BULK_STAGES 4
#endif
#ifndef RESHARD_BULK_CHUNK
#define RESHARD_BULK_CHUNK 49152
#endif
constexpr int kBulkStages = RESHARD_BULK_STAGES;
constexpr int kBulkChunk = RESHARD_BULK_CHUNK;  // bytes per stage (multiple of 16)
constexpr size_t kBulkSmem = (size_t)kBulkStages * kBulkChunk;

__device__ __forceinline__ bool bulk_wait(uint32_t bar, uint32_t parity) {
  const unsigned long long deadline = global_ns() + kWaitLimitNs;
  return bar_wait(bar, parity, deadline);
}

struct BulkPiece {
  const uint8_t *src;
  int64_t dst_off;  // bytes from each member's item base
  int len;
};

__global__ void __launch_bounds__(32, 1) reshard_bulk_kernel(const Item *__restrict__ items,
                                                             const int32_t *__restrict__ idx, int n_items,
                                                             const uint64_t *__restrict__ ptrs,
                                                             const int32_t *__restrict__ gstart,
                                                             const int32_t *__restrict__ mptr,
                                                             const int64_t *__restrict__ moff, int32_t *status) {
  pdl_enter();
  extern __shared__ __align__(128) uint8_t bulk_buf[];
  __shared__ __align__(8) uint64_t bar[kBulkStages];
  if (threadIdx.x != 0) return;
  for (int s = 0; s < kBulkStages; ++s) asm volatile("mbarrier.init.shared::cta.b64 [%0], 1;" ::"r"(smem_u32(&bar[s])));
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");

  // piece cursor over this CTA's items: item k, row r, byte offset c within the row
  int k = blockIdx.x, r = 0;
  int64_t c = 0;
  Item it{};
  if (k < n_items) it = items[item_index(idx, k)];
  auto next_piece = [&](BulkPiece &pc, Item &owner) -> bool {
    while (k < n_items) {
      const int64_t run_b = (int64_t)it.run * it.esize;
      if (r < it.rows && c < run_b) {
        pc.src = reinterpret_cast<const uint8_t *>(ptrs[it.src]) + (it.src_off + r * it.src_pitch) * it.esize + c;
        pc.dst_off = (it.dst_off + (int64_t)r * it.dst_pitch) * it.esize + c;
        pc.len = (int)(run_b - c < kBulkChunk ? run_b - c : (int64_t)kBulkChunk);
        owner = it;
        c += pc.len;
        if (c >= run_b) {
          c = 0;
          ++r;
        }
        return true;
      }
      k += gridDim.x;
      r = 0;
      c = 0;
      if (k < n_items) it = items[item_index(idx, k)];
    }
    return false;
  };

  BulkPiece ring[kBulkStages];
  Item owner[kBulkStages];
  uint32_t phases = 0;
  int issued = 0;  // pieces whose load was issued
  auto issue_load = [&](int stage) -> bool {
    if (!next_piece(ring[stage], owner[stage])) return false;
    const uint32_t b = smem_u32(&bar[stage]);
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(b), "r"(ring[stage].len) : "memory");
    asm volatile("cp.async.bulk.shared::cta.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
                     smem_u32(bulk_buf + (size_t)stage * kBulkChunk)),
                 "l"(ring[stage].src), "r"(ring[stage].len), "r"(b)
                 : "memory");
    ++issued;
    return true;
  };
  int loaded = 0;
  for (int s = 0; s < kBulkStages - 1; ++s)
    if (issue_load(s)) ++loaded;
  for (int t = 0; t < loaded; ++t) {
    const int stage = t % kBulkStages;
    if (!bulk_wait(smem_u32(&bar[stage]), (phases >> stage) & 1)) {
      // a load never completed: report, give every load in flight one more bounded wait, stop
      atomicOr(status, 1);
      for (int u = t; u < loaded; ++u) {
        const int su = u % kBulkStages;
        bulk_wait(smem_u32(&bar[su]), (phases >> su) & 1);
      }
      break;
    }
    phases ^= 1u << stage;
    const Item &o = owner[stage];
    const int g0 = gstart[o.group], g1 = gstart[o.group + 1];
    for (int m = g0; m < g1; ++m) {
      uint8_t *d = reinterpret_cast<uint8_t *>(ptrs[mptr[m]]) + moff[m] * o.esize + ring[stage].dst_off;
      asm volatile("cp.async.bulk.global.shared::cta.bulk_group [%0], [%1], %2;" ::"l"(d),
                   "r"(smem_u32(bulk_buf + (size_t)stage * kBulkChunk)), "r"(ring[stage].len)
                   : "memory");
    }
    asm volatile("cp.async.bulk.commit_group;" ::: "memory");
    // reload the stage the previous piece's stores were reading, once they are done reading it
    const int next_stage = (t + kBulkStages - 1) % kBulkStages;
    asm volatile("cp.async.bulk.wait_group.read 1;" ::: "memory");
    if (issue_load(next_stage)) ++loaded;
  }
  asm volatile("cp.async.bulk.wait_group 0;" ::: "memory");
}

// ---------------------------------------------------------------------------- host side --

namespace {

int cuda_fail(cudaError_t e, const char *what) {
  return fail(e == cudaErrorMemoryAllocation ? RESHARD_ERR_OOM : RESHARD_ERR_CUDA,
              std::string(what) + ": " + cudaGetErrorString(e));
}

#define RS_CUDA(call)                                   \
  do {                                                  \
    cudaError_t e_ = (call);                            \
    if (e_ != cudaSuccess) return cuda_fail(e_, #call); \
  } while (0)

template <typename T>
int upload(T **dptr, const std::vector<T> &host) {
  if (host.empty()) return RESHARD_OK;
  RS_CUDA(cudaMalloc(reinterpret_cast<void **>(dptr), host.size() * sizeof(T)));
  RS_CUDA(cudaMemcpy(*dptr, host.data(), host.size() * sizeof(T), cudaMemcpyHostToDevice));
  return RESHARD_OK;
}

// Launch with programmatic stream serialization allowed when `pdl` (the kernels begin with
// pdl_enter). The transposing kernel is launched without: measured 0.4-1.5% slower with it.
template <typename... KArgs, typename... Args>
cudaError_t launch_kernel(bool pdl, void (*kernel)(KArgs...), int grid, int block, size_t smem, cudaStream_t stream,
                          Args &&...args) {
  cudaLaunchConfig_t cfg{};
  cfg.gridDim = dim3((unsigned)grid);
  cfg.blockDim = dim3((unsigned)block);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = RESHARD_PDL && pdl ? 1 : 0;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kernel, std::forward<Args>(args)...);
}

struct LaunchCaps {
  int device = -1;
  int bulk_grid = 0;
  int aligned_grid = 0;
  int copy_grid = 0;
  int rows_grid = 0;
  int gather_grid = 0;
  int scatter_grid = 0;
  int staged_grid = 0;
  int mxfp8_grid = 0;
  int transpose_grid[4] = {0, 0, 0, 0};  // per element size 1, 2, 4, 8 bytes
};
thread_local LaunchCaps g_caps;

int launch_caps(int device, LaunchCaps &c) {
  if (g_caps.device == device) {
    c = g_caps;
    return RESHARD_OK;
  }
  int sms = 0, b0 = 0, b1 = 0, b2 = 0, b4 = 0;
  RS_CUDA(cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, device));
  RS_CUDA(cudaOccupancyMaxActiveBlocksPerMultiprocessor(&b0, reshard_copy_aligned_kernel, kBlock, 0));
  int bb = 0;
  if (RESHARD_BULK) {
    RS_CUDA(cudaFuncSetAttribute(reshard_bulk_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kBulkSmem));
    RS_CUDA(cudaOccupancyMaxActiveBlocksPerMultiprocessor(&bb, reshard_bulk_kernel, 32, kBulkSmem));
  }
  RS_CUDA(cudaOccupancyMaxActiveBlocksPerMultiprocessor(&b1, reshard_copy_kernel, kBlock, 0));
  RS_CUDA(cudaOccupancyMaxActiveBlocksPerMultiprocessor(&b4, reshard_copy_rows_kernel, kBlock, 0));
  int bg = 0, bsc = 0;
  RS_CUDA(cudaOccupancyMaxActiveBlocksPerMultiprocessor(&bg, reshard_copy_gather_kernel, kBlock, 0));
  RS_CUDA(cudaOccupancyMaxActiveBlocksPerMultiprocessor(&bsc, reshard_copy_scatter_kernel, kBlock, 0));
  int bs = 0;
  RS_CUDA(cudaFuncSetAttribute(reshard_copy_staged_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kStagedSmem));
  RS_CUDA(cudaOccupancyMaxActiveBlocksPerMultiprocessor(&bs, reshard_copy_staged_kernel, kBlock, kStagedSmem));
  RS_CUDA(cudaOccupancyMaxActiveBlocksPerMultiprocessor(&b2, reshard_mxfp8_kernel, kQBlock, 0));
  int bt[4] = {0, 0, 0, 0};
  RS_CUDA(cudaOccupancyMaxActiveBlocksPerMultiprocessor(&bt[0], reshard_transpose_kernel<1>, kTBlock, 0));
  RS_CUDA(cudaOccupancyMaxActiveBlocksPerMultiprocessor(&bt[1], reshard_transpose_kernel<2>, kTBlock, 0));
  RS_CUDA(cudaOccupancyMaxActiveBlocksPerMultiprocessor(&bt[2], reshard_transpose_kernel<4>, kTBlock, 0));
  RS_CUDA(cudaOccupancyMaxActiveBlocksPerMultiprocessor(&bt[3], reshard_transpose_kernel<8>, kTBlock, 0));
  g_caps.device = device;
  g_caps.aligned_grid = sms * std::max(1, b0);
  g_caps.bulk_grid = sms * std::max(1, bb);
  g_caps.copy_grid = sms * std::max(1, b1);
  g_caps.rows_grid = sms * std::max(1, b4);
  g_caps.gather_grid = sms * std::max(1, bg);
  g_caps.scatter_grid = sms * std::max(1, bsc);
  g_caps.staged_grid = sms * std::max(1, bs);
  g_caps.mxfp8_grid = sms * std::max(1, b2);
  for (int k = 0; k < 4; ++k) g_caps.transpose_grid[k] = sms * std::max(1, bt[k]);
  c = g_caps;
  return RESHARD_OK;
}

int bind_device(reshard_plan_t *p) {
  int dev = 0;
  RS_CUDA(cudaGetDevice(&dev));
  if (p->device >= 0) {
    if (dev != p->device)
      return fail(RESHARD_ERR_INVALID_ARG, "plan was bound to device " + std::to_string(p->device) +
                                               " by its first execute; current device is " + std::to_string(dev));
    return RESHARD_OK;
  }
  int rc;
  if ((rc = upload(&p->d_grp_start, p->grp_start))) return rc;
  if ((rc = upload(&p->d_mem_ptr, p->mem_ptr))) return rc;
  if ((rc = upload(&p->d_mem_off, p->mem_off))) return rc;
  RS_CUDA(cudaMalloc(reinterpret_cast<void **>(&p->d_ptrs), pointer_table_size(p) * sizeof(uint64_t)));
  RS_CUDA(cudaMalloc(reinterpret_cast<void **>(&p->d_status), sizeof(int32_t)));
  RS_CUDA(cudaMemset(p->d_status, 0, sizeof(int32_t)));
  if (!p->slabs.empty()) {
    RS_CUDA(cudaMalloc(&p->d_maps, p->slabs.size() * sizeof(CUtensorMap)));
    RS_CUDA(cudaMalloc(reinterpret_cast<void **>(&p->d_map_ok), p->slabs.size() * sizeof(int32_t)));
  }
  p->device = dev;
  return RESHARD_OK;
}

// cuTensorMapEncodeTiled from the driver, looked up once through the runtime.
std::once_flag g_encode_once;
PFN_cuTensorMapEncodeTiled_v12000 g_encode = nullptr;

PFN_cuTensorMapEncodeTiled_v12000 tensor_map_encoder() {
  std::call_once(g_encode_once, [] {
    void *fn = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      g_encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
  });
  return g_encode;
}

// Every pointer the kernels dereference must be reachable from `device`: memory of that device,
// managed memory, or page-locked host memory mapped into the device's address space
// (cudaHostAlloc, cudaMallocHost, cudaHostRegister). The kernels then read and write host memory
// in place over the host link. A host pointer whose device alias differs from it is replaced by
// the alias in `*dev`; `*host` marks host memory, over which no TMA tensor map is encoded.
// Returns why the entry is refused, or nullptr (NULL entries are never dereferenced and pass).
const char *check_entry(int device, uint64_t v, uint64_t *dev, uint8_t *host) {
  *dev = v;
  *host = 0;
  if (!v) return nullptr;
  cudaPointerAttributes a{};
  if (cudaPointerGetAttributes(&a, reinterpret_cast<const void *>(v)) != cudaSuccess) {
    (void)cudaGetLastError();
    a.type = cudaMemoryTypeUnregistered;
  }
  if (a.type == cudaMemoryTypeDevice) return a.device != device ? "is memory of another device" : nullptr;
  if (a.type == cudaMemoryTypeHost) {
    if (!a.devicePointer) return "is page-locked host memory without a device mapping";
    *dev = reinterpret_cast<uint64_t>(a.devicePointer);
    *host = 1;
    return nullptr;
  }
  if (a.type == cudaMemoryTypeManaged) return nullptr;
  return "is pageable host memory (page-lock it with cudaHostRegister or use device memory)";
}

std::string entry_name(int64_t i, int64_t Ns, int64_t Nd) {
  return i < Ns            ? "source pointer " + std::to_string(i)
         : i < Ns + Nd     ? "destination pointer " + std::to_string(i - Ns)
         : i < Ns + 2 * Nd ? "scale pointer " + std::to_string(i - Ns - Nd)
         : i == Ns + 2 * Nd ? std::string("send buffer")
                            : std::string("receive buffer");
}

// One 2-D tensor map per source slab of the transposing items, for the current pointers. A slab
// whose base or row pitch is not 16-byte aligned (or that the driver rejects) gets map_ok = 0:
// its tiles are then loaded with plain loads.
int encode_maps(reshard_plan_t *p, const std::vector<uint64_t> &table, const std::vector<uint8_t> &host,
                cudaStream_t stream) {
  const size_t n = p->slabs.size();
  if (!n) return RESHARD_OK;
  std::vector<CUtensorMap> maps(n);
  std::vector<int32_t> ok(n, 0);
  PFN_cuTensorMapEncodeTiled_v12000 enc = tensor_map_encoder();
  for (size_t i = 0; i < n && enc; ++i) {
    const SlabSpec &sl = p->slabs[i];
    const uint64_t base = table[(size_t)sl.ptr] + (uint64_t)sl.base_off * (uint64_t)sl.esize;
    const uint64_t stride = (uint64_t)sl.pitch * (uint64_t)sl.esize;
    if (!table[(size_t)sl.ptr] || host[(size_t)sl.ptr] || base % 16 || stride % 16 || stride == 0 || stride >= (1ull << 40) || sl.cols < 1 ||
        sl.rows < 1 || sl.cols > (1ll << 32) || sl.rows > (1ll << 32))
      continue;
    const CUtensorMapDataType dt = sl.esize == 1   ? CU_TENSOR_MAP_DATA_TYPE_UINT8
                                   : sl.esize == 2 ? CU_TENSOR_MAP_DATA_TYPE_UINT16
                                   : sl.esize == 4 ? CU_TENSOR_MAP_DATA_TYPE_UINT32
                                                   : CU_TENSOR_MAP_DATA_TYPE_UINT64;
    const cuuint64_t dims[2] = {(cuuint64_t)sl.cols, (cuuint64_t)sl.rows};
    const cuuint64_t strides[1] = {stride};
    const cuuint32_t box[2] = {(cuuint32_t)(kTileRowBytes / sl.esize), (cuuint32_t)kTileRows};
    const cuuint32_t estr[2] = {1, 1};
    const CUresult r = enc(&maps[i], dt, 2, reinterpret_cast<void *>(base), dims, strides, box, estr,
                           CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_128B,
                           CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    ok[i] = r == CUDA_SUCCESS ? 1 : 0;
  }
  RS_CUDA(cudaMemcpyAsync(p->d_maps, maps.data(), n * sizeof(CUtensorMap), cudaMemcpyHostToDevice, stream));
  RS_CUDA(cudaMemcpyAsync(p->d_map_ok, ok.data(), n * sizeof(int32_t), cudaMemcpyHostToDevice, stream));
  return RESHARD_OK;
}

int ensure_items(reshard_plan_t *p, int set) {
  if (p->d_items[set] || p->items[set].empty()) return RESHARD_OK;
  Item *d = nullptr;
  int rc = upload(&d, p->items[set]);
  p->d_items[set] = d;
  return rc;
}

int launch_transpose(reshard_plan_t *p, int set, cudaStream_t stream, const LaunchCaps &caps) {
  const int n = (int)p->titems[set].size();
  if (n == 0) return RESHARD_OK;
  if (!p->d_titems[set]) {
    TItem *d = nullptr;
    int rc = upload(&d, p->titems[set]);
    p->d_titems[set] = d;
    if (rc) return rc;
  }
  // the planner sorted the items by element size: one launch per run of equal sizes
  const std::vector<TItem> &tv = p->titems[set];
  const TItem *d_items = static_cast<const TItem *>(p->d_titems[set]);
  const CUtensorMap *maps = static_cast<const CUtensorMap *>(p->d_maps);
  for (int b = 0; b < n;) {
    cudaError_t rc = cudaSuccess;
    const int es = tv[(size_t)b].esize;
    int e = b;
    while (e < n && tv[(size_t)e].esize == es) ++e;
    const int k = es == 1 ? 0 : es == 2 ? 1 : es == 4 ? 2 : 3;
    const int grid = std::min(e - b, caps.transpose_grid[k]);
    const TItem *items = d_items + b;
    switch (es) {
      case 1:
        rc = launch_kernel(false, reshard_transpose_kernel<1>, grid, kTBlock, 0, stream, items, e - b, p->d_ptrs,
                           p->d_grp_start, p->d_mem_ptr, p->d_mem_off, maps, p->d_map_ok, p->d_status);
        break;
      case 2:
        rc = launch_kernel(false, reshard_transpose_kernel<2>, grid, kTBlock, 0, stream, items, e - b, p->d_ptrs,
                           p->d_grp_start, p->d_mem_ptr, p->d_mem_off, maps, p->d_map_ok, p->d_status);
        break;
      case 4:
        rc = launch_kernel(false, reshard_transpose_kernel<4>, grid, kTBlock, 0, stream, items, e - b, p->d_ptrs,
                           p->d_grp_start, p->d_mem_ptr, p->d_mem_off, maps, p->d_map_ok, p->d_status);
        break;
      default:
        rc = launch_kernel(false, reshard_transpose_kernel<8>, grid, kTBlock, 0, stream, items, e - b, p->d_ptrs,
                           p->d_grp_start, p->d_mem_ptr, p->d_mem_off, maps, p->d_map_ok, p->d_status);
        break;
    }
    if (rc != cudaSuccess) return cuda_fail(rc, "launching reshard_transpose_kernel");
    ++p->last_launches;
    b = e;
  }
  return RESHARD_OK;
}

// Split the copy items of `set` into those 16-byte aligned everywhere for the current pointers
// (source, every replica, run, pitches) and the rest; upload the order on `stream`.
int classify(reshard_plan_t *p, int set, cudaStream_t stream) {
  if (p->cls_version[set] == p->ptr_version && (p->d_cls_idx[set] || p->cls_idx[set].empty())) return RESHARD_OK;
  const std::vector<Item> &items = p->items[set];
  const std::vector<uint64_t> &tab = p->dev_ptrs;
  std::vector<int32_t> &idx = p->cls_idx[set];
  idx.clear();
  idx.reserve(items.size());
  std::vector<int32_t> staged, general;
  int64_t gen_bytes = 0, row_bytes = 0;
  // bulk copies read device memory only (page-locked host memory goes through the walkers)
  const bool stage_ok = RESHARD_STAGED && !p->any_host;
  // the pass's gather items write the rows of the copy items flagged kGathered
  const bool gathered = !p->gitems[set].empty();
  for (size_t i = 0; i < items.size(); ++i) {
    const Item &it = items[i];
    if (gathered && it.pad[0] == kGathered) continue;
    const uint64_t es = (uint64_t)it.esize;
    uint64_t m = tab[(size_t)it.src] + (uint64_t)it.src_off * es;
    m |= (uint64_t)it.run * es;
    if (it.rows > 1) m |= (uint64_t)it.src_pitch * es | (uint64_t)it.dst_pitch * es;
    for (int32_t k = p->grp_start[(size_t)it.group]; k < p->grp_start[(size_t)it.group + 1]; ++k)
      m |= tab[(size_t)p->mem_ptr[(size_t)k]] + (uint64_t)(p->mem_off[(size_t)k] + it.dst_off) * es;
    const int64_t run_b = (int64_t)it.run * (int64_t)es;
    if ((m & 15) == 0) {
      idx.push_back((int32_t)i);
    } else if (stage_ok && it.rows > 1 && run_b <= kStagedMaxRun &&
               p->grp_start[(size_t)it.group + 1] - p->grp_start[(size_t)it.group] <= kStagedFan) {
      staged.push_back((int32_t)i);
    } else {
      general.push_back((int32_t)i);
      const int64_t b = (int64_t)it.rows * run_b;
      gen_bytes += b;
      if (it.rows > 1 && run_b < RESHARD_ROWS_MAX_RUN) row_bytes += b;
    }
  }
  // Short single-replica launches go to the many-rows walker instead: there its 48 resident
  // warps start faster than the staged kernel's 16 warp pipelines fill (measured at 117 MB of
  // rows: 0.716 against 0.684 of the copy rate), while with two or more replicas, or at 4x the
  // bytes, staging wins (0.731 against 0.709; 0.735 against 0.709).
  if (!staged.empty()) {
    int64_t traffic = 0;
    int max_rep = 0;
    for (int32_t i : staged) {
      const Item &it = items[(size_t)i];
      const int nrep = p->grp_start[(size_t)it.group + 1] - p->grp_start[(size_t)it.group];
      traffic += (int64_t)it.rows * it.run * it.esize * (1 + nrep);
      max_rep = std::max(max_rep, nrep);
    }
    if (max_rep < 2 && traffic < kStagedMinTraffic) {
      for (int32_t i : staged) {
        const Item &it = items[(size_t)i];
        const int64_t b = (int64_t)it.rows * it.run * it.esize;
        gen_bytes += b;
        if ((int64_t)it.run * it.esize < RESHARD_ROWS_MAX_RUN) row_bytes += b;
      }
      general.insert(general.begin(), staged.begin(), staged.end());
      staged.clear();
    }
  }
  p->n_aligned[set] = (int32_t)idx.size();
  p->n_staged[set] = (int32_t)staged.size();
  p->n_general[set] = (int32_t)general.size();
  // the general items run in the many-rows build when most of their bytes are short rows
  p->gen_rows[set] = 2 * row_bytes > gen_bytes;
  idx.insert(idx.end(), staged.begin(), staged.end());
  idx.insert(idx.end(), general.begin(), general.end());
  if (!p->d_cls_idx[set] && !idx.empty())
    RS_CUDA(cudaMalloc(reinterpret_cast<void **>(&p->d_cls_idx[set]), idx.size() * sizeof(int32_t)));
  if (!idx.empty())
    RS_CUDA(cudaMemcpyAsync(p->d_cls_idx[set], idx.data(), idx.size() * sizeof(int32_t), cudaMemcpyHostToDevice,
                            stream));
  p->cls_version[set] = p->ptr_version;
  return RESHARD_OK;
}

// Resolve the gather items of pass `set` for the current pointer table (absolute addresses of both
// pieces and of the first two replicas) and upload them on `stream`, when the table has changed.
int bind_gather(reshard_plan_t *p, int set, cudaStream_t stream) {
  if (p->d_gbound[set] && p->gbound_version[set] == p->ptr_version) return RESHARD_OK;
  const std::vector<uint64_t> &tab = p->dev_ptrs;
  const size_t n = p->gitems[set].size();
  std::vector<GBound> &bound = p->gbound[set];
  bound.resize(n);
  for (size_t i = 0; i < n; ++i) {
    const GItem &g = p->gitems[set][i];
    GBound &b = bound[i];
    const uint64_t es = (uint64_t)g.esize;
    const int32_t m0 = p->grp_start[(size_t)g.group];
    const int32_t nrep = p->grp_start[(size_t)g.group + 1] - m0;
    for (int k = 0; k < 2; ++k) {
      b.src[k] = tab[(size_t)g.src[k]] + (uint64_t)g.src_off[k] * es;
      b.sp[k] = g.src_pitch[k] * (int64_t)es;
    }
    for (int f = 0; f < 2; ++f) {
      if (g.kind == kScatterRow) {  // piece f's row 0 in the group's one member (the send buffer)
        b.dst[f] = tab[(size_t)p->mem_ptr[(size_t)m0]] + (uint64_t)(p->mem_off[(size_t)m0] + g.dst_off[f]) * es;
      } else {                      // row 0 in replica f
        const int32_t m = m0 + (f < nrep ? f : 0);
        b.dst[f] = tab[(size_t)p->mem_ptr[(size_t)m]] + (uint64_t)(p->mem_off[(size_t)m] + g.dst_off[0]) * es;
      }
      b.dp[f] = g.dst_pitch[f] * (int64_t)es;
    }
    b.dst_off_b = g.dst_off[0] * (int64_t)es;
    b.B = g.run[0] * g.esize;
    b.rb = b.B + g.run[1] * g.esize;
    b.rows = g.rows;
    b.group = g.group;
    b.nrep = nrep;
    b.esize = g.esize;
    b.kind = g.kind;
    b.pad = 0;
  }
  if (!p->d_gbound[set]) RS_CUDA(cudaMalloc(&p->d_gbound[set], n * sizeof(GBound)));
  RS_CUDA(cudaMemcpyAsync(p->d_gbound[set], bound.data(), n * sizeof(GBound), cudaMemcpyHostToDevice, stream));
  p->gbound_version[set] = p->ptr_version;
  return RESHARD_OK;
}

int launch(reshard_plan_t *p, int set, bool quant, cudaStream_t stream, const LaunchCaps &caps) {
  int rc = launch_transpose(p, set, stream, caps);  // counts its own launches
  if (rc) return rc;
  const int n = (int)p->items[set].size();
  if (n == 0) return RESHARD_OK;
  rc = ensure_items(p, set);
  if (rc) return rc;
  const Item *items = static_cast<const Item *>(p->d_items[set]);
  if (quant) {
    const int grid = std::min(n, caps.mxfp8_grid);
    RS_CUDA(launch_kernel(true, reshard_mxfp8_kernel, grid, kQBlock, 0, stream, items, n, p->d_ptrs, p->d_grp_start,
                          p->d_mem_ptr, p->d_mem_off, p->n_dst_ptrs));
    ++p->last_launches;
  } else {
    if ((rc = classify(p, set, stream))) return rc;
    const int na = p->n_aligned[set], ns = p->n_staged[set], ng = p->n_general[set];
    const int nx = (int)p->gitems[set].size();
    const int32_t *idx = p->d_cls_idx[set];
    p->last_aligned = na;
    p->last_staged = ns;
    p->last_general = ng;
    p->last_gather += nx;
    if (na > 0 && RESHARD_BULK && !p->any_host) {  // bulk copies over device memory only
      RS_CUDA(launch_kernel(true, reshard_bulk_kernel, std::min(na, caps.bulk_grid), 32, kBulkSmem, stream, items, idx, na,
                            p->d_ptrs, p->d_grp_start, p->d_mem_ptr, p->d_mem_off, p->d_status));
      ++p->last_launches;
    } else if (na > 0) {
      RS_CUDA(launch_kernel(true, reshard_copy_aligned_kernel, std::min(na, caps.aligned_grid), kBlock, 0, stream, items,
                            idx, na, p->d_ptrs, p->d_grp_start, p->d_mem_ptr, p->d_mem_off, p->d_status));
      ++p->last_launches;
    }
    p->last_rows_kernel = ng > 0 && p->gen_rows[set];
    // a later launch of the pass starts while the earlier ones drain (their items touch other
    // bytes) and takes its dependency wait just before it exits
    if (ns > 0) {
      const int wait_last = RESHARD_GEN_OVERLAP && na > 0 ? 1 : 0;
      RS_CUDA(launch_kernel(true, reshard_copy_staged_kernel, std::min(ns, caps.staged_grid), kBlock, kStagedSmem, stream,
                            items, idx + na, ns, p->d_ptrs, p->d_grp_start, p->d_mem_ptr, p->d_mem_off, p->d_status,
                            wait_last));
      ++p->last_launches;
    }
    const int wait_last = RESHARD_GEN_OVERLAP && na + ns > 0 ? 1 : 0;
    if (ng > 0 && p->gen_rows[set]) {
      RS_CUDA(launch_kernel(true, reshard_copy_rows_kernel, std::min(ng, caps.rows_grid), kBlock, 0, stream, items,
                            idx + na + ns, ng, p->d_ptrs, p->d_grp_start, p->d_mem_ptr, p->d_mem_off, wait_last));
      ++p->last_launches;
    } else if (ng > 0) {
      RS_CUDA(launch_kernel(true, reshard_copy_kernel, std::min(ng, caps.copy_grid), kBlock, 0, stream, items,
                            idx + na + ns, ng, p->d_ptrs, p->d_grp_start, p->d_mem_ptr, p->d_mem_off, wait_last));
      ++p->last_launches;
    }
    if (nx > 0) {
      if ((rc = bind_gather(p, set, stream))) return rc;
      const int wait_gather = RESHARD_GEN_OVERLAP && na + ns + ng > 0 ? 1 : 0;
      const GBound *gb = static_cast<const GBound *>(p->d_gbound[set]);
      if (set == kPack)
        RS_CUDA(launch_kernel(true, reshard_copy_scatter_kernel, std::min(nx, caps.scatter_grid), kBlock, 0, stream, gb,
                              nx, wait_gather));
      else
        RS_CUDA(launch_kernel(true, reshard_copy_gather_kernel, std::min(nx, caps.gather_grid), kBlock, 0, stream, gb,
                              nx, p->d_ptrs, p->d_grp_start, p->d_mem_ptr, p->d_mem_off, wait_gather));
      ++p->last_launches;
    }
  }
  RS_CUDA(cudaGetLastError());
  return RESHARD_OK;
}

void free_device(reshard_plan_t *p) {
  for (auto &d : p->d_items) {
    if (d) cudaFree(d);
    d = nullptr;
  }
  for (auto &d : p->d_titems) {
    if (d) cudaFree(d);
    d = nullptr;
  }
  for (auto &d : p->d_cls_idx) {
    if (d) cudaFree(d);
    d = nullptr;
  }
  for (auto &d : p->d_gbound) {
    if (d) cudaFree(d);
    d = nullptr;
  }
  if (p->d_maps) cudaFree(p->d_maps);
  if (p->d_map_ok) cudaFree(p->d_map_ok);
  if (p->d_status) cudaFree(p->d_status);
  p->d_maps = nullptr;
  p->d_map_ok = nullptr;
  p->d_status = nullptr;
  if (p->d_grp_start) cudaFree(p->d_grp_start);
  if (p->d_mem_ptr) cudaFree(p->d_mem_ptr);
  if (p->d_mem_off) cudaFree(p->d_mem_off);
  if (p->d_ptrs) cudaFree(p->d_ptrs);
  if (p->d_workspace) cudaFree(p->d_workspace);
  p->d_grp_start = nullptr;
  p->d_mem_ptr = nullptr;
  p->d_mem_off = nullptr;
  p->d_ptrs = nullptr;
  p->d_workspace = nullptr;
}

}  // namespace
}  // namespace reshard

using namespace reshard;

namespace reshard {
namespace {

// Entries of the pointer table that one call provides: (index, caller's value).
typedef std::vector<std::pair<int64_t, uint64_t>> PtrUpdate;

void provide_sources(const reshard_plan_t *p, void *const *src_ptrs, PtrUpdate &u) {
  for (int64_t i = 0; i < p->n_src_ptrs; ++i) u.emplace_back(i, reinterpret_cast<uint64_t>(src_ptrs[i]));
}

void provide_destinations(const reshard_plan_t *p, void *const *dst_ptrs, bool quant, PtrUpdate &u) {
  const int64_t Ns = p->n_src_ptrs, Nd = p->n_dst_ptrs;
  for (int64_t i = 0; i < Nd; ++i) {
    u.emplace_back(Ns + i, reinterpret_cast<uint64_t>(quant ? dst_ptrs[2 * i] : dst_ptrs[i]));
    u.emplace_back(Ns + Nd + i, quant ? reinterpret_cast<uint64_t>(dst_ptrs[2 * i + 1]) : 0);
  }
}

// Every entry the passes `sets` dereference is non-NULL in `u` (scales too under quant).
int check_used(const reshard_plan_t *p, const PtrUpdate &u, std::initializer_list<int> sets, bool quant) {
  const int64_t Ns = p->n_src_ptrs, Nd = p->n_dst_ptrs;
  std::vector<uint64_t> val((size_t)pointer_table_size(p), 0);
  std::vector<char> given((size_t)pointer_table_size(p), 0);
  for (const auto &e : u) {
    val[(size_t)e.first] = e.second;
    given[(size_t)e.first] = 1;
  }
  std::string missing;
  int n = 0;
  auto need = [&](int64_t i) {
    if ((!given[(size_t)i] || !val[(size_t)i]) && n++ < 8) missing += "\n  " + entry_name(i, Ns, Nd) + " is NULL";
  };
  for (int set : sets) {
    for (int32_t i : p->used_src[set]) need(i);
    for (int32_t i : p->used_dst[set]) {
      need(i);
      if (quant && set != kPack) need(i + Nd);
    }
  }
  if (n) return fail(RESHARD_ERR_INVALID_ARG, std::to_string(n) + " NULL pointer(s) the kernels need:" + missing);
  return RESHARD_OK;
}

// Bring the device pointer table up to date with the entries this call provides (entries it
// does not provide keep their values; the passes it runs do not read them). Changed entries are
// checked first, so a refused pointer leaves the table as it was.
int stage_pointers(reshard_plan_t *p, const PtrUpdate &u, cudaStream_t stream) {
  const size_t n = (size_t)pointer_table_size(p);
  if (p->ptr_cache.size() != n) {
    p->ptr_cache.assign(n, 0);
    p->dev_ptrs.assign(n, 0);
    p->ptr_host.assign(n, 0);
    p->ptr_cache_valid = false;
  }
  const int64_t Ns = p->n_src_ptrs, Nd = p->n_dst_ptrs;
  std::vector<std::pair<int64_t, std::pair<uint64_t, uint8_t>>> changed;
  std::string bad;
  int n_bad = 0;
  for (const auto &e : u) {
    if (p->ptr_cache_valid && p->ptr_cache[(size_t)e.first] == e.second) continue;
    uint64_t dv;
    uint8_t host;
    const char *why = check_entry(p->device, e.second, &dv, &host);
    if (why) {
      if (n_bad++ < 8) {
        char addr[32];
        std::snprintf(addr, sizeof addr, "0x%llx", (unsigned long long)e.second);
        bad += "\n  " + entry_name(e.first, Ns, Nd) + " (" + addr + ") " + why;
      }
      continue;
    }
    changed.emplace_back(e.first, std::make_pair(dv, host));
  }
  if (n_bad) return fail(RESHARD_ERR_INVALID_ARG, std::to_string(n_bad) + " pointer(s) the device cannot dereference:" + bad);
  if (changed.empty() && p->ptr_cache_valid) return RESHARD_OK;
  for (const auto &e : u) p->ptr_cache[(size_t)e.first] = e.second;
  for (const auto &c : changed) {
    p->dev_ptrs[(size_t)c.first] = c.second.first;
    p->ptr_host[(size_t)c.first] = c.second.second;
  }
  // pageable source: the runtime stages the bytes before returning, so the table may change
  RS_CUDA(cudaMemcpyAsync(p->d_ptrs, p->dev_ptrs.data(), n * sizeof(uint64_t), cudaMemcpyHostToDevice, stream));
  int rc = encode_maps(p, p->dev_ptrs, p->ptr_host, stream);
  if (rc) return rc;
  p->any_host = std::find(p->ptr_host.begin(), p->ptr_host.end(), 1) != p->ptr_host.end();
  ++p->ptr_version;
  p->ptr_cache_valid = true;
  return RESHARD_OK;
}

// Completion of this call's work on `stream`, for destroy to wait on (not under stream capture:
// a captured execute runs when its graph is replayed, and the plan must outlive the graph).
void record_done(reshard_plan_t *p, cudaStream_t stream) {
  cudaStreamCaptureStatus cs = cudaStreamCaptureStatusNone;
  if (cudaStreamIsCapturing(stream, &cs) != cudaSuccess) {
    (void)cudaGetLastError();
    return;
  }
  if (cs != cudaStreamCaptureStatusNone) return;
  for (auto &e : p->done_events)
    if (e.first == static_cast<void *>(stream)) {
      cudaEventRecord(static_cast<cudaEvent_t>(e.second), stream);
      return;
    }
  // forget streams whose last execute has finished, then track this one
  for (size_t i = 0; i < p->done_events.size();) {
    cudaEvent_t ev = static_cast<cudaEvent_t>(p->done_events[i].second);
    if (cudaEventQuery(ev) == cudaSuccess) {
      cudaEventDestroy(ev);
      p->done_events.erase(p->done_events.begin() + (long)i);
    } else {
      (void)cudaGetLastError();
      ++i;
    }
  }
  cudaEvent_t ev = nullptr;
  if (cudaEventCreateWithFlags(&ev, cudaEventDisableTiming) != cudaSuccess) {
    (void)cudaGetLastError();
    return;
  }
  cudaEventRecord(ev, stream);
  p->done_events.emplace_back(static_cast<void *>(stream), static_cast<void *>(ev));
}

int check_mode_quant(const reshard_plan_t *p, int quant) {
  if (quant != RESHARD_QUANT_NONE && quant != RESHARD_QUANT_MXFP8) return fail(RESHARD_ERR_INVALID_ARG, "unknown quant");
  if (quant == RESHARD_QUANT_MXFP8 && !p->quant_ok) return fail(RESHARD_ERR_UNSUPPORTED, p->quant_why);
  return RESHARD_OK;
}

int check_message_buffer(const reshard_plan_t *p, const void *buf, int64_t bytes, const char *what) {
  if (bytes <= 0) return RESHARD_OK;
  if (!buf) return fail(RESHARD_ERR_INVALID_ARG, std::string(what) + " is NULL");
  if (reinterpret_cast<uintptr_t>(buf) & 15) return fail(RESHARD_ERR_INVALID_ARG, std::string(what) + " is not 16-byte aligned");
  (void)p;
  return RESHARD_OK;
}

}  // namespace
}  // namespace reshard

extern "C" int reshard_execute(reshard_plan_t *p, void *const *src_ptrs, void *const *dst_ptrs, int mode, int quant,
                               reshard_stream_t stream_) {
  if (!p) return fail(RESHARD_ERR_INVALID_ARG, "plan is NULL");
  if (p->rank >= 0)
    return fail(RESHARD_ERR_INVALID_ARG, "a partitioned plan runs through reshard_execute_pack and reshard_execute_unpack");
  if (mode != RESHARD_DIRECT && mode != RESHARD_PACKED) return fail(RESHARD_ERR_INVALID_ARG, "unknown mode");
  int rc = check_mode_quant(p, quant);
  if (rc) return rc;
  if (p->regions.empty()) return RESHARD_OK;
  if ((p->n_src_ptrs && !src_ptrs) || (p->n_dst_ptrs && !dst_ptrs))
    return fail(RESHARD_ERR_INVALID_ARG, "src_ptrs or dst_ptrs is NULL");
  cudaStream_t stream = reinterpret_cast<cudaStream_t>(stream_);
  const bool q = quant == RESHARD_QUANT_MXFP8;
  PtrUpdate u;
  provide_sources(p, src_ptrs, u);
  provide_destinations(p, dst_ptrs, q, u);
  if (mode == RESHARD_DIRECT) {
    if ((rc = check_used(p, u, {kDirect}, q))) return rc;
  } else if ((rc = check_used(p, u, {kPack, kUnpack}, q))) {
    return rc;
  }
  if ((rc = bind_device(p))) return rc;
  LaunchCaps caps;
  if ((rc = launch_caps(p->device, caps))) return rc;
  if (mode == RESHARD_PACKED) {
    if (!p->d_workspace && p->stats.message_bytes > 0) RS_CUDA(cudaMalloc(&p->d_workspace, (size_t)p->stats.message_bytes));
    u.emplace_back(p->workspace_ptr, reinterpret_cast<uint64_t>(p->d_workspace));
    u.emplace_back(p->workspace_ptr + 1, reinterpret_cast<uint64_t>(p->d_workspace));
  }
  if ((rc = stage_pointers(p, u, stream))) return rc;
  p->last_launches = 0;
  p->last_gather = 0;
  if (mode == RESHARD_DIRECT) {
    rc = launch(p, kDirect, q, stream, caps);
  } else if (!(rc = launch(p, kPack, false, stream, caps))) {
    rc = launch(p, kUnpack, q, stream, caps);
  }
  if (!rc) record_done(p, stream);
  return rc;
}

extern "C" int reshard_execute_pack(reshard_plan_t *p, void *const *src_ptrs, void *const *dst_ptrs, void *send_buf,
                                    int quant, reshard_stream_t stream_) {
  if (!p) return fail(RESHARD_ERR_INVALID_ARG, "plan is NULL");
  int rc = check_mode_quant(p, quant);
  if (rc) return rc;
  const bool q = quant == RESHARD_QUANT_MXFP8;
  if (p->rank < 0 && q) return fail(RESHARD_ERR_INVALID_ARG, "packing an unpartitioned plan does not quantize");
  // an unpartitioned plan's direct table is reshard_execute's; only a partition's is local copies
  const bool direct = p->rank >= 0 && (!p->items[kDirect].empty() || !p->titems[kDirect].empty());
  const bool pack = !p->items[kPack].empty() || !p->titems[kPack].empty();
  if (!direct && !pack) return RESHARD_OK;
  if (p->n_src_ptrs && !src_ptrs) return fail(RESHARD_ERR_INVALID_ARG, "src_ptrs is NULL");
  if (direct && p->n_dst_ptrs && !dst_ptrs) return fail(RESHARD_ERR_INVALID_ARG, "dst_ptrs is NULL");
  if (pack && (rc = check_message_buffer(p, send_buf, p->stats.message_bytes, "send_buf"))) return rc;
  cudaStream_t stream = reinterpret_cast<cudaStream_t>(stream_);
  PtrUpdate u;
  provide_sources(p, src_ptrs, u);
  if (dst_ptrs) provide_destinations(p, dst_ptrs, q, u);
  if ((rc = direct ? check_used(p, u, {kDirect, kPack}, q) : check_used(p, u, {kPack}, q))) return rc;
  if ((rc = bind_device(p))) return rc;
  LaunchCaps caps;
  if ((rc = launch_caps(p->device, caps))) return rc;
  u.emplace_back(p->workspace_ptr, reinterpret_cast<uint64_t>(send_buf));
  if ((rc = stage_pointers(p, u, stream))) return rc;
  p->last_launches = 0;
  p->last_gather = 0;
  if (direct && (rc = launch(p, kDirect, q, stream, caps))) return rc;
  if (pack && (rc = launch(p, kPack, false, stream, caps))) return rc;
  record_done(p, stream);
  return RESHARD_OK;
}

extern "C" int reshard_execute_unpack(reshard_plan_t *p, const void *recv_buf, void *const *dst_ptrs, int quant,
                                      reshard_stream_t stream_) {
  if (!p) return fail(RESHARD_ERR_INVALID_ARG, "plan is NULL");
  int rc = check_mode_quant(p, quant);
  if (rc) return rc;
  if (p->items[kUnpack].empty() && p->titems[kUnpack].empty()) return RESHARD_OK;
  if (p->n_dst_ptrs && !dst_ptrs) return fail(RESHARD_ERR_INVALID_ARG, "dst_ptrs is NULL");
  if ((rc = check_message_buffer(p, recv_buf, p->stats.recv_bytes, "recv_buf"))) return rc;
  const bool q = quant == RESHARD_QUANT_MXFP8;
  cudaStream_t stream = reinterpret_cast<cudaStream_t>(stream_);
  PtrUpdate u;
  provide_destinations(p, dst_ptrs, q, u);
  if ((rc = check_used(p, u, {kUnpack}, q))) return rc;
  if ((rc = bind_device(p))) return rc;
  LaunchCaps caps;
  if ((rc = launch_caps(p->device, caps))) return rc;
  u.emplace_back(p->workspace_ptr + 1, reinterpret_cast<uint64_t>(recv_buf));
  if ((rc = stage_pointers(p, u, stream))) return rc;
  p->last_launches = 0;
  p->last_gather = 0;
  if ((rc = launch(p, kUnpack, q, stream, caps))) return rc;
  record_done(p, stream);
  return RESHARD_OK;
}

extern "C" int reshard_plan_status(reshard_plan_t *p, int32_t *status, int reset) {
  if (!p || !status) return fail(RESHARD_ERR_INVALID_ARG, "plan or status is NULL");
  *status = 0;
  if (p->device < 0 || !p->d_status) return RESHARD_OK;
  int cur = 0;
  RS_CUDA(cudaGetDevice(&cur));
  RS_CUDA(cudaSetDevice(p->device));
  cudaError_t e = cudaDeviceSynchronize();
  if (e == cudaSuccess) e = cudaMemcpy(status, p->d_status, sizeof(int32_t), cudaMemcpyDeviceToHost);
  if (e == cudaSuccess && reset) e = cudaMemset(p->d_status, 0, sizeof(int32_t));
  cudaSetDevice(cur);
  if (e != cudaSuccess) return cuda_fail(e, "reading the plan status");
  return RESHARD_OK;
}

extern "C" int reshard_plan_destroy(reshard_plan_t *p) {
  if (!p) return RESHARD_OK;
  if (p->device >= 0) {
    int cur = 0;
    cudaGetDevice(&cur);
    cudaSetDevice(p->device);
    // Executes of this plan may still be queued (a garbage-collected handle, for instance): wait
    // for the last one on every stream it used, not for the whole device. Relaxed capture mode
    // keeps these waits and frees from invalidating a stream capture another thread runs.
    cudaStreamCaptureMode mode = cudaStreamCaptureModeRelaxed;
    const bool swapped = cudaThreadExchangeStreamCaptureMode(&mode) == cudaSuccess;
    for (auto &e : p->done_events) {
      cudaEvent_t ev = static_cast<cudaEvent_t>(e.second);
      cudaEventSynchronize(ev);
      cudaEventDestroy(ev);
    }
    p->done_events.clear();
    free_device(p);
    if (swapped) cudaThreadExchangeStreamCaptureMode(&mode);
    (void)cudaGetLastError();
    cudaSetDevice(cur);
  }
  delete p;
  return RESHARD_OK;
}

// ------------------------------------------------------------ execute without allocating --
//
// Some callers must not have a library allocate device memory on their behalf. A generation
// engine that has reserved almost all of the GPU for its KV cache, or a framework whose own
// caching allocator owns the device heap, cannot let a weight refit call cudaMalloc: the call
// can fail for lack of memory, and cudaMalloc / cudaFree synchronize the device and would stall
// generation. reshard_execute_static serves them: it runs the direct-mode copy with its
// descriptor tables held in the file-scope array below, which is part of the library image and
// is reserved once on every GPU that loads the library, for as long as the process lives.

// Every call uses this one array and it keeps the previous call's contents; nothing in it has to
// start at zero (the kernel reads only what the current call copied in). Calls that overlap on
// the GPU (different streams, or other threads) overwrite each other's tables and race.
static __device__ __align__(256) unsigned char reshard_static_scratch[RESHARD_STATIC_SCRATCH_BYTES];

namespace reshard {
namespace {

constexpr int kMaxDevices = 64;
std::mutex g_static_mu;
uint8_t *g_static_addr[kMaxDevices] = {};
// the pointers of the last call on each device that passed the reachability check (host memory)
struct StaticCheck {
  std::vector<uint64_t> given, dev;
};
StaticCheck g_static_check[kMaxDevices];

// Device address of the scratch array on device `dev` (which must be current). The host-side
// name of a __device__ array is not a device address, so it is looked up once per device with
// cudaGetSymbolAddress on the first call made there.
int static_scratch(int dev, uint8_t **out) {
  if (dev < 0 || dev >= kMaxDevices) return fail(RESHARD_ERR_UNSUPPORTED, "device ordinal above 63");
  std::lock_guard<std::mutex> lock(g_static_mu);
  if (!g_static_addr[dev]) {
    void *p = nullptr;
    cudaError_t e = cudaGetSymbolAddress(&p, reshard_static_scratch);
    if (e != cudaSuccess) return cuda_fail(e, "cudaGetSymbolAddress(reshard_static_scratch)");
    g_static_addr[dev] = static_cast<uint8_t *>(p);
  }
  *out = g_static_addr[dev];
  return RESHARD_OK;
}

size_t align256(size_t x) { return (x + 255) / 256 * 256; }

}  // namespace
}  // namespace reshard

extern "C" int reshard_execute_static(const reshard_plan_t *p, void *const *src_ptrs, void *const *dst_ptrs,
                                      reshard_stream_t stream_) {
  using namespace reshard;
  if (!p) return fail(RESHARD_ERR_INVALID_ARG, "plan is NULL");
  if (p->rank >= 0)
    return fail(RESHARD_ERR_INVALID_ARG, "a partitioned plan runs through reshard_execute_pack and reshard_execute_unpack");
  if (!p->titems[kDirect].empty())
    return fail(RESHARD_ERR_UNSUPPORTED, "plans with transposing regions need reshard_execute (TMA tensor maps)");
  // scratch layout: items | group starts | member pointers | member offsets | pointer table
  const std::vector<Item> &items = p->items[kDirect];
  const size_t b_items = items.size() * sizeof(Item);
  const size_t b_gs = p->grp_start.size() * sizeof(int32_t);
  const size_t b_mp = p->mem_ptr.size() * sizeof(int32_t);
  const size_t b_mo = p->mem_off.size() * sizeof(int64_t);
  const size_t b_pt = (size_t)pointer_table_size(p) * sizeof(uint64_t);
  const size_t o_gs = align256(b_items), o_mp = o_gs + align256(b_gs), o_mo = o_mp + align256(b_mp);
  const size_t o_pt = o_mo + align256(b_mo), need = o_pt + align256(b_pt);
  if (need > (size_t)RESHARD_STATIC_SCRATCH_BYTES)
    return fail(RESHARD_ERR_UNSUPPORTED, "plan needs " + std::to_string(need) +
                                             " bytes of descriptor scratch; reshard_execute_static holds at most " +
                                             std::to_string((size_t)RESHARD_STATIC_SCRATCH_BYTES) +
                                             " (split the batch or use reshard_execute)");
  if (!p->regions.empty() && ((p->n_src_ptrs && !src_ptrs) || (p->n_dst_ptrs && !dst_ptrs)))
    return fail(RESHARD_ERR_INVALID_ARG, "src_ptrs or dst_ptrs is NULL");
  PtrUpdate u;
  if (!p->regions.empty()) {
    provide_sources(p, src_ptrs, u);
    for (int64_t i = 0; i < p->n_dst_ptrs; ++i)
      u.emplace_back(p->n_src_ptrs + i, reinterpret_cast<uint64_t>(dst_ptrs[i]));
    int rc = check_used(p, u, {kDirect}, false);
    if (rc) return rc;
  }
  // set-up on every call, an empty plan's too: the array's device address on this device (the
  // lookup loads the library's device code here, which reserves the array)
  int dev = 0;
  RS_CUDA(cudaGetDevice(&dev));
  uint8_t *base = nullptr;
  int rc = static_scratch(dev, &base);
  if (rc) return rc;
  if (p->regions.empty()) return RESHARD_OK;
  // the pointers the kernel will dereference must be reachable from this device, as for
  // reshard_execute; the last validated table (per device) is remembered, so repeated calls with
  // the same pointers skip the per-pointer queries
  std::vector<uint64_t> table((size_t)pointer_table_size(p), 0);
  {
    std::lock_guard<std::mutex> lock(g_static_mu);
    std::vector<uint64_t> given((size_t)(p->n_src_ptrs + p->n_dst_ptrs));
    for (size_t k = 0; k < given.size(); ++k) given[k] = u[k].second;
    StaticCheck &c = g_static_check[dev];
    if (c.given != given) {
      std::string bad;
      int n_bad = 0;
      std::vector<uint64_t> devp(given.size());
      for (size_t k = 0; k < given.size(); ++k) {
        uint8_t host;
        const char *why = check_entry(dev, given[k], &devp[k], &host);
        if (why && n_bad++ < 8) {
          char addr[32];
          std::snprintf(addr, sizeof addr, "0x%llx", (unsigned long long)given[k]);
          bad += "\n  " + entry_name((int64_t)k, p->n_src_ptrs, p->n_dst_ptrs) + " (" + addr + ") " + why;
        }
      }
      if (n_bad)
        return fail(RESHARD_ERR_INVALID_ARG, std::to_string(n_bad) + " pointer(s) the device cannot dereference:" + bad);
      c.given = std::move(given);
      c.dev = std::move(devp);
    }
    std::copy(c.dev.begin(), c.dev.end(), table.begin());
  }
  LaunchCaps caps;
  if ((rc = launch_caps(dev, caps))) return rc;
  cudaStream_t stream = reinterpret_cast<cudaStream_t>(stream_);
  // pageable sources: the runtime stages them before each call returns
  RS_CUDA(cudaMemcpyAsync(base, items.data(), b_items, cudaMemcpyHostToDevice, stream));
  RS_CUDA(cudaMemcpyAsync(base + o_gs, p->grp_start.data(), b_gs, cudaMemcpyHostToDevice, stream));
  RS_CUDA(cudaMemcpyAsync(base + o_mp, p->mem_ptr.data(), b_mp, cudaMemcpyHostToDevice, stream));
  RS_CUDA(cudaMemcpyAsync(base + o_mo, p->mem_off.data(), b_mo, cudaMemcpyHostToDevice, stream));
  // pointer table [sources | destinations | ...]: the direct copy reads only these two runs
  RS_CUDA(cudaMemcpyAsync(base + o_pt, table.data(), (size_t)(p->n_src_ptrs + p->n_dst_ptrs) * sizeof(uint64_t),
                          cudaMemcpyHostToDevice, stream));
  const int n = (int)items.size();
  const int grid = std::min(n, caps.copy_grid);
  reshard_copy_kernel<<<grid, kBlock, 0, stream>>>(
      reinterpret_cast<const Item *>(base), nullptr, n, reinterpret_cast<const uint64_t *>(base + o_pt),
      reinterpret_cast<const int32_t *>(base + o_gs), reinterpret_cast<const int32_t *>(base + o_mp),
      reinterpret_cast<const int64_t *>(base + o_mo), 0);
  RS_CUDA(cudaGetLastError());
  return RESHARD_OK;
}
