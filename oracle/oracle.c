/*
 * Reshard oracle in plain scalar C. TEST INFRASTRUCTURE: only the tests, the package entry's
 * smoke check and the bench's CPU-baseline leg load this library. It shares no code with the
 * CUDA path (no headers, helpers or tables in common).
 *
 * It writes out the golden semantics of the debugging transport in the NeMo-RL design doc
 * "NCCL Reshard Refit (Experimental)", section "xferdtensor Transports": the full tensor is
 * rebuilt from the source shards and every destination keeps its own slice. With quant = 1
 * each destination shard is then quantized to MXFP8 ("Enabling It": generation ranks
 * quantize each received BF16 shard), by the OCP MX v1.0 block rule with OFP8 E4M3 elements.
 *
 * Readings (also in the design notes): torch.chunk's uneven split (chunk = ceil(L / n));
 * nested mesh dims split in mesh-dim order; row-major rank numbering; an all-zero MXFP8 block
 * gets scale byte 0x00; a block holding Inf/NaN gets scale 0xFF and elements 0x7F.
 *
 * Parity: cross-checked against the Python oracle (which is pinned by the 8x8 worked example,
 * brute force and torch.chunk) and, for MXFP8, against brute-force nearest-code enumeration
 * over every BF16 pattern; the placement of a quantized shard (E4M3 bytes row-major from the
 * shard's element offset, E8M0 scales row-major [..., K_local / 32] from offset / 32) against a
 * hand-derived fixture whose every scale byte and code block names its block, and against the
 * Python oracle's independent placement (tests). Single-threaded; one tensor per call.
 */
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#define ORACLE_MAX_DIMS 8

enum { ORACLE_OK = 0, ORACLE_REPLICA_MISMATCH = 1, ORACLE_UNCOVERED = 2, ORACLE_BAD_ARGS = 3,
       ORACLE_NO_MEMORY = 4 };

/* torch.chunk rule: chunk size ceil(L / n); piece i is [min(i c, L), min((i + 1) c, L)). */
static void chunk_bounds(int64_t len, int64_t n, int64_t i, int64_t *lo, int64_t *hi) {
    int64_t c = len > 0 ? (len + n - 1) / n : 0;
    int64_t a = i * c, b = (i + 1) * c;
    *lo = a < len ? a : len;
    *hi = b < len ? b : len;
}

/* Box of the rank whose row-major mesh position is `rank`. placement[k] < 0: Replicate,
 * otherwise Shard(placement[k]). Mesh dims are applied in order (nested chunking). */
static void shard_box(int nd, const int64_t *gshape, int md, const int64_t *mesh,
                      const int32_t *placement, int64_t rank, int64_t *lo, int64_t *hi) {
    int64_t coord[ORACLE_MAX_DIMS];
    for (int k = md - 1; k >= 0; --k) {
        coord[k] = rank % mesh[k];
        rank /= mesh[k];
    }
    for (int d = 0; d < nd; ++d) {
        lo[d] = 0;
        hi[d] = gshape[d];
    }
    for (int k = 0; k < md; ++k) {
        int d = placement[k];
        if (d < 0) continue;
        int64_t a, b;
        chunk_bounds(hi[d] - lo[d], mesh[k], coord[k], &a, &b);
        hi[d] = lo[d] + b;
        lo[d] = lo[d] + a;
    }
}

static int64_t prod(int n, const int64_t *v) {
    int64_t p = 1;
    for (int i = 0; i < n; ++i) p *= v[i];
    return p;
}

/* Element strides of a view: given ones, or dense row-major of the local shape. */
static void view_strides(int nd, const int64_t *shape, const int64_t *given, int64_t *out) {
    if (given) {
        for (int d = 0; d < nd; ++d) out[d] = given[d];
        return;
    }
    int64_t s = 1;
    for (int d = nd - 1; d >= 0; --d) {
        out[d] = s;
        s *= shape[d];
    }
}

/* Advance a multi-index over the outer dims [0, nd-1) of `ext`; returns 0 when done. */
static int next_outer(int nd, const int64_t *ext, int64_t *idx) {
    for (int d = nd - 2; d >= 0; --d) {
        if (++idx[d] < ext[d]) return 1;
        idx[d] = 0;
    }
    return 0;
}

/* ---------------------------------------------------------------- MXFP8 (OCP MX v1.0) -- */

/* floor(log2 |v|) of a finite nonzero BF16 magnitude (bits without sign). */
static int bf16_floor_log2(uint32_t mag) {
    uint32_t e = mag >> 7;
    if (e) return (int)e - 127;
    int p = 31 - __builtin_clz(mag);  /* subnormal: value = m * 2^-133 */
    return -133 + p;
}

/* |v| = M * 2^E with integer M for a finite BF16 magnitude. */
static void bf16_split(uint32_t mag, int64_t *M, int *E) {
    uint32_t e = mag >> 7, m = mag & 0x7F;
    if (e) {
        *M = 128 + m;
        *E = (int)e - 127 - 7;
    } else {
        *M = m;
        *E = -133;
    }
}

/* E4M3 code of (M * 2^E) / 2^X, round to nearest even, saturating at 448; sign bit `s`. */
uint8_t oracle_e4m3(uint16_t bits, int x) {
    uint8_t s = (bits >> 15) ? 0x80 : 0x00;
    uint32_t mag = bits & 0x7FFF;
    if (mag == 0) return s;
    int64_t M;
    int E;
    bf16_split(mag, &M, &E);
    E -= x;                                  /* |q| = M * 2^E exactly */
    int lg = bf16_floor_log2(mag) - x;       /* floor(log2 |q|) */
    int qe = lg >= -6 ? lg - 3 : -9;         /* quantum exponent: 3 mantissa bits, or 2^-9 */
    int sh = E - qe;                         /* |q| / quantum = M * 2^sh */
    int64_t k;
    if (sh >= 0) {
        k = sh > 20 ? ((int64_t)1 << 40) : (M << sh);
    } else {
        int r = -sh;
        if (r > 20) {
            k = 0;                           /* M < 2^8, far below half a quantum */
        } else {
            int64_t q = M >> r, rem = M & (((int64_t)1 << r) - 1), half = (int64_t)1 << (r - 1);
            k = q + ((rem > half || (rem == half && (q & 1))) ? 1 : 0);
        }
    }
    /* the rounded value is k * 2^qe; anything above 448 saturates to 448 */
    if (k == 0) return s;
    {
        int over;
        if (qe >= 0) over = qe > 20 || (k << qe) > 448;
        else over = qe < -40 ? 0 : (k > ((int64_t)448 << (-qe)));
        if (over) return s | 0x7E;          /* 448 = 1.75 * 2^8: exponent field 15, mantissa 6 */
    }
    /* encode k * 2^qe */
    if (qe == -9 && k < 8) return s | (uint8_t)k;          /* subnormal m * 2^-9 */
    /* normal: bring k into [8, 16) */
    while (k >= 16) {                        /* only k == 16 after a carry */
        k >>= 1;
        qe += 1;
    }
    while (k < 8) {                          /* subnormal range rounded up to 2^-6 */
        k <<= 1;
        qe -= 1;
    }
    int e_field = qe + 3 + 7;
    return s | (uint8_t)((e_field << 3) | (k - 8));
}

/* Shared exponent of a block of 32 BF16 values: X, or 128 when the block holds Inf/NaN. */
int oracle_block_exponent(const uint16_t *v) {
    uint32_t amax = 0;
    for (int i = 0; i < 32; ++i) {
        uint32_t mag = v[i] & 0x7FFF;
        if (mag >= 0x7F80) return 128;
        if (mag > amax) amax = mag;
    }
    if (amax == 0) return -127;
    int x = bf16_floor_log2(amax) - 8;       /* 8 = exponent of E4M3's largest normal */
    if (x < -127) x = -127;
    if (x > 127) x = 127;
    return x;
}

void oracle_mxfp8_block(const uint16_t *v, uint8_t *out, uint8_t *scale) {
    int x = oracle_block_exponent(v);
    if (x == 128) {
        for (int i = 0; i < 32; ++i) out[i] = 0x7F;
        *scale = 0xFF;
        return;
    }
    for (int i = 0; i < 32; ++i) out[i] = oracle_e4m3(v[i], x);
    *scale = (uint8_t)(x + 127);
}

/* ------------------------------------------------------------------- golden reshard -- */

/*
 * One tensor. Buffers are raw host byte pointers, one per rank (row-major mesh order).
 * Views: element offset per rank, element strides per rank (n_ranks * nd values) or NULL
 * for dense row-major of the local shape. quant = 1: destination buffers receive E4M3 bytes
 * and d_scales the E8M0 bytes (dense views only; offset and last local dim multiples of 32).
 */
int oracle_reshard_tensor(int nd, const int64_t *gshape, int esize,
                          int s_md, const int64_t *s_mesh, const int32_t *s_pl,
                          const uint8_t *const *s_bufs, const int64_t *s_off, const int64_t *s_strides,
                          int d_md, const int64_t *d_mesh, const int32_t *d_pl,
                          uint8_t *const *d_bufs, const int64_t *d_off, const int64_t *d_strides,
                          int quant, uint8_t *const *d_scales) {
    if (nd < 1 || nd > ORACLE_MAX_DIMS || s_md < 1 || s_md > ORACLE_MAX_DIMS || d_md < 1 ||
        d_md > ORACLE_MAX_DIMS)
        return ORACLE_BAD_ARGS;
    if (quant && (esize != 2 || d_strides)) return ORACLE_BAD_ARGS;
    int64_t numel = prod(nd, gshape);
    int64_t gstr[ORACLE_MAX_DIMS];
    view_strides(nd, gshape, NULL, gstr);
    uint8_t *full = (uint8_t *)malloc((size_t)(numel ? numel : 1) * esize);
    uint8_t *have = (uint8_t *)calloc((size_t)(numel ? numel : 1), 1);
    if (!full || !have) {
        free(full);
        free(have);
        return ORACLE_NO_MEMORY;
    }
    int rc = ORACLE_OK;
    int64_t lo[ORACLE_MAX_DIMS], hi[ORACLE_MAX_DIMS], ext[ORACLE_MAX_DIMS], st[ORACLE_MAX_DIMS],
        idx[ORACLE_MAX_DIMS];

    /* 1. rebuild the full tensor from every source shard, checking replicas agree */
    int64_t n_src = prod(s_md, s_mesh);
    for (int64_t r = 0; r < n_src && rc == ORACLE_OK; ++r) {
        shard_box(nd, gshape, s_md, s_mesh, s_pl, r, lo, hi);
        for (int d = 0; d < nd; ++d) ext[d] = hi[d] - lo[d];
        if (prod(nd, ext) == 0) continue;
        view_strides(nd, ext, s_strides ? s_strides + r * nd : NULL, st);
        memset(idx, 0, sizeof(idx));
        do {
            int64_t g0 = lo[nd - 1], l0 = s_off[r];
            for (int d = 0; d < nd - 1; ++d) {
                g0 += (lo[d] + idx[d]) * gstr[d];
                l0 += idx[d] * st[d];
            }
            for (int64_t j = 0; j < ext[nd - 1] && rc == ORACLE_OK; ++j) {
                int64_t g = g0 + j, l = l0 + j * st[nd - 1];
                const uint8_t *src = s_bufs[r] + l * esize;
                if (have[g]) {
                    if (memcmp(full + g * esize, src, esize)) rc = ORACLE_REPLICA_MISMATCH;
                } else {
                    memcpy(full + g * esize, src, esize);
                    have[g] = 1;
                }
            }
        } while (rc == ORACLE_OK && next_outer(nd, ext, idx));
    }
    for (int64_t g = 0; g < numel && rc == ORACLE_OK; ++g)
        if (!have[g]) rc = ORACLE_UNCOVERED;

    /* 2. every destination keeps its own slice (quantized under quant = 1) */
    int64_t n_dst = prod(d_md, d_mesh);
    for (int64_t r = 0; r < n_dst && rc == ORACLE_OK; ++r) {
        shard_box(nd, gshape, d_md, d_mesh, d_pl, r, lo, hi);
        for (int d = 0; d < nd; ++d) ext[d] = hi[d] - lo[d];
        if (prod(nd, ext) == 0) continue;
        if (quant && (ext[nd - 1] % 32 || d_off[r] % 32)) {
            rc = ORACLE_BAD_ARGS;
            break;
        }
        view_strides(nd, ext, d_strides ? d_strides + r * nd : NULL, st);
        memset(idx, 0, sizeof(idx));
        int64_t row = 0;
        do {
            int64_t g0 = 0, l0 = d_off[r];
            for (int d = 0; d < nd - 1; ++d) {
                g0 += (lo[d] + idx[d]) * gstr[d];
                l0 += idx[d] * st[d];
            }
            g0 += lo[nd - 1];
            if (!quant) {
                for (int64_t j = 0; j < ext[nd - 1]; ++j)
                    memcpy(d_bufs[r] + (l0 + j * st[nd - 1]) * esize, full + (g0 + j) * esize, esize);
            } else {
                int64_t nb = ext[nd - 1] / 32;
                for (int64_t b = 0; b < nb; ++b) {
                    uint16_t blk[32];
                    memcpy(blk, full + (g0 + 32 * b) * 2, 64);
                    oracle_mxfp8_block(blk, d_bufs[r] + l0 + 32 * b,
                                       d_scales[r] + d_off[r] / 32 + row * nb + b);
                }
            }
            ++row;
        } while (next_outer(nd, ext, idx));
    }
    free(full);
    free(have);
    return rc;
}
