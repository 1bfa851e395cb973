// Row-grouped GEMM on tcgen05 with warp-specialised roles (k_umma2).
//
// The contraction and epilogue of k_umma (moe_umma.cuh), with the three jobs
// of a 64-column K-chunk in different warps that meet on mbarriers, so that
// copies, int4 dequantisation and tensor-core MMAs of different chunks
// overlap.  Work units are (group, 128-row A tile, token tile); every operand
// tile is K-major with the 128-byte swizzle.
//
//   warps 1-3  producers: the copies of ring slot q (SUB = 1 or 2 chunks).
//              Thread 0 issues tensor copies against host-encoded maps: the
//              A operand (16-bit weight rows, or int4 codes and their
//              group-major scale/bias words) and, where the rows form a
//              plain matrix, the B operand (the dense tokens, or the pairs'
//              rows in sorted order), and arrives on full[s] with their byte
//              count.  What no map describes goes by cp.async from all 96
//              threads, each arriving through cp.async.mbarrier.arrive.noinc
//              when its copies land; no producer waits for its own copies,
//              and with every operand by tensor copies thread 0 is the only
//              producer.  (A per-thread wait for landed copies before
//              arriving tied the ring to the MMAs two chunks back.)
//   warps 4-7  dequant: int4 -> 16-bit A tile in buffer c % NA (after full[s]
//              and after the MMAs of chunk c - NA released the buffer), then
//              arrive on dfull[c % NA].  After a tile's last chunk they read
//              the accumulators from tensor memory and write the epilogue.
//   warp 0     lane 0 issues the tcgen05.mma of chunk c once dfull[c % NA]
//              completes and commits them to dempty[c % NA] (the A buffer may
//              be rewritten), after a slot's last chunk to empty[s] (the slot
//              may be refilled) and after a tile's last chunk to acc (the
//              accumulators are final).
//
// Every role walks the same sequence of tiles, slots and chunks, so the
// barrier phases are implied by the counts.  Every wait is bounded (waiting
// roles sleep between polls); on a timeout the role sets the status word's
// timeout bit and stops, the other roles' waits then run out too, and the
// kernel drains its copies and MMAs (bounded) before it frees tensor memory.
#pragma once

#include "moe_umma.cuh"

namespace moe {

// Byte offset of element (row, k) of a 64-column 16-bit tile in the 128-byte
// swizzled K-major layout (row r's 128 bytes at r * 128, its 16-byte piece j
// at position j ^ (r & 7)); the tile starts on a 1024-byte boundary.
__device__ __forceinline__ uint32_t sw_off(int row, int k) {
  return static_cast<uint32_t>(row * 128 + ((((k >> 3) ^ row) & 7) << 4) + (k & 7) * 2);
}

// Eight int4 codes (one word, code i in bits 4i..4i+3) -> s*q + b as four
// words of two 16-bit values (codes 2i, 2i+1 in word i), s2 / b2 the scale
// and bias in both halves.  A code becomes the 16-bit number M + q by filling
// the low mantissa bits of M (128 in bf16, 1024 in fp16, exact for q < 16);
// subtracting M is exact and one packed fma rounds s*q + b once to the type.
// Codes i and i + 4 share a word until the byte permutes put pairs in order.
__device__ __forceinline__ void dq8_packed(uint32_t v, uint32_t s2, uint32_t b2, int dt, uint32_t (&o)[4]) {
  const uint32_t magic = dt == DT_BF16 ? 0x43004300u : 0x64006400u;
  uint32_t y[4];
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const uint32_t x = ((v >> (4 * i)) & 0x000F000Fu) | magic;
    if (dt == DT_BF16) {
      const __nv_bfloat162 r = __hfma2(__hsub2(*reinterpret_cast<const __nv_bfloat162*>(&x),
                                               *reinterpret_cast<const __nv_bfloat162*>(&magic)),
                                       *reinterpret_cast<const __nv_bfloat162*>(&s2),
                                       *reinterpret_cast<const __nv_bfloat162*>(&b2));
      y[i] = *reinterpret_cast<const uint32_t*>(&r);
    } else {
      const __half2 r = __hfma2(__hsub2(*reinterpret_cast<const __half2*>(&x),
                                        *reinterpret_cast<const __half2*>(&magic)),
                                *reinterpret_cast<const __half2*>(&s2), *reinterpret_cast<const __half2*>(&b2));
      y[i] = *reinterpret_cast<const uint32_t*>(&r);
    }
  }
  o[0] = __byte_perm(y[0], y[1], 0x5410);
  o[1] = __byte_perm(y[2], y[3], 0x5410);
  o[2] = __byte_perm(y[0], y[1], 0x7632);
  o[3] = __byte_perm(y[2], y[3], 0x7632);
}

// B pieces (16 bytes) a producer thread copies per chunk: 96 producers, up to
// 128 tokens x 8 pieces
constexpr int UM_BPIECES = (128 * 8 + 95) / 96;

// One unit's tile: rows [m0, m_end) of A (dense: inside segment si), the
// group's tokens [n0, n0 + nvalid) padded to npad, K-chunks [kc_begin, + nit).
struct UmmaTile {
  int split, kc_begin, nit, n0, nvalid, npad, si, m0, m_end;
  UmmaGroup G;
};

__device__ __forceinline__ void mbar_arrive(uint32_t mbar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(mbar) : "memory");
}

__global__ void __launch_bounds__(UM_THREADS, 2) k_umma2(const __grid_constant__ UmmaArgs A) {
  extern __shared__ __align__(1024) char um_smem[];
  const bool gated = (A.a_mode == UA_INT4) && A.q2 != nullptr;
  const int SUB = A.sub > 1 ? 2 : 1;   // 64-column chunks per ring slot
  const UmmaPlan P = umma_plan(A.a_mode, gated, A.n_tile, A.stages, A.abufs, SUB, A.G);
  const uint32_t CB = P.code_bytes, SBB = P.sb_bytes;
  const int NA = A.abufs;   // dequantised A tiles: chunk c uses buffer c % NA
  // the plan starts on a 1024-byte boundary (swizzled tiles; the plan has the room)
  char* base = um_smem + ((1024u - (smem_u32(um_smem) & 1023u)) & 1023u);
  const bool tma = A.tma_a != 0;
  // every operand by tensor copies: thread 0 alone produces (no cp.async arrivals)
  const bool all_tma = tma && A.tma_b != 0;
  const int S = A.stages;
  // barriers and the tensor-memory address in the plan's token-table area
  uint64_t* bars = reinterpret_cast<uint64_t*>(base + P.tok);
  uint64_t* full = bars;               // [S]  producers' copies landed (96 arrivals)
  uint64_t* empty = bars + S;          // [S]  MMAs of the slot's chunk done (commit)
  uint64_t* dfull = bars + 2 * S;      // [NA] A tile ready (128 arrivals)
  uint64_t* dempty = dfull + NA;       // [NA] MMAs reading the A tile done (commit)
  uint64_t* accb = dempty + NA;        // [1]  a tile's accumulators final (commit)
  uint64_t* epib = accb + 1;           // [1]  the epilogue has read them (128 arrivals)
  uint64_t* drainb = epib + 1;         // [1]  every MMA issued has completed (final commit)
  uint32_t* tmem_holder = reinterpret_cast<uint32_t*>(drainb + 1);
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int ncols = gated ? 512 : 256;
  // diagnostics: role stamps of CTA 0 -- producer thread 0: 0 (before the slot
  // wait), 1 (slot free), 2 (transaction bytes announced), 3 (first tensor
  // copy issued), 4 (all tensor copies issued), 11 (cp.async copies issued),
  // 10 (cp.async arrival done); dequant 5 (copies landed), 6 (A buffer free),
  // 7 (done); MMA 8 (start), 9 (issued)
  unsigned long long* const trace = (A.trace && blockIdx.x == 0) ? A.trace : nullptr;
  // (SM cycle counter: exact within the CTA)
  auto stamp = [&](uint32_t chunk, int k) {
    if (trace && chunk < static_cast<uint32_t>(UM_TRACE_CHUNKS)) trace[chunk * UM_TRACE_STAMPS + k] = clock64();
  };
  if (trace && tid == 0) trace[UM_TRACE_CHUNKS * UM_TRACE_STAMPS] = clock64();

  griddep_wait();
  griddep_launch();
  if (warp == 0) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                     smem_u32(tmem_holder)),
                 "r"(ncols));
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;");
  }
  if (tid == 0) {
    for (int s = 0; s < S; ++s) {
      mbar_init(smem_u32(&full[s]), all_tma ? 1 : ((tma || A.tma_b) ? 97 : 96));
      mbar_init(smem_u32(&empty[s]), 1);
    }
    for (int b = 0; b < NA; ++b) {
      mbar_init(smem_u32(&dfull[b]), 128);
      mbar_init(smem_u32(&dempty[b]), 1);
    }
    mbar_init(smem_u32(accb), 1);
    mbar_init(smem_u32(epib), 128);
    mbar_init(smem_u32(drainb), 1);
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  const int n_groups = A.experts ? A.meta[0] : 1;
  int* pref = reinterpret_cast<int*>(base + P.pref);
  tc_fence_before();
  umma_tile_prefix(A, n_groups, pref, pref + UM_MAX_GROUPS + 1);   // ends with a CTA barrier
  tc_fence_after();
  const uint32_t tmem = *tmem_holder;

  // 128-row tiles of A: an expert's rows from 0; a dense matrix's per
  // segment, so that no tile crosses a segment (a segment's last tile is
  // partial) and a chunk of A is one tensor copy
  int mtiles = (A.n_rows + UM_M - 1) / UM_M;
  if (!A.experts) {
    mtiles = 0;
    for (int si = 0; si < A.nseg; ++si) mtiles += (A.seg[si].rows + UM_M - 1) / UM_M;
  }
  const int nkc = A.K / UM_KC;
  const int ngr = A.K / A.G;
  const int nsplit = A.ksplit > 1 ? A.ksplit : 1;
  const int nunits = pref[n_groups] * mtiles * nsplit;
  bool ok = true;

  // Walk the units of this CTA: fn(tile)
  auto tiles = [&](auto&& fn) {
    for (int unit = blockIdx.x; ok && unit < nunits; unit += gridDim.x) {
      const UmmaUnit U = umma_unit(pref, n_groups, mtiles, nsplit, unit);
      UmmaTile Tl;
      Tl.split = U.split;
      Tl.kc_begin = static_cast<int>(static_cast<int64_t>(U.split) * nkc / nsplit);
      Tl.nit = static_cast<int>(static_cast<int64_t>(U.split + 1) * nkc / nsplit) - Tl.kc_begin;
      Tl.G = umma_group(A, U.g);
      Tl.n0 = U.nt * A.n_tile;
      Tl.nvalid = min(A.n_tile, Tl.G.n - Tl.n0);
      Tl.npad = (Tl.nvalid + 15) & ~15;
      if (A.experts) {
        Tl.si = 0;
        Tl.m0 = U.mt * UM_M;
        Tl.m_end = A.n_rows;
      } else {
        int mt = U.mt, si = 0;
        while (mt >= (A.seg[si].rows + UM_M - 1) / UM_M) mt -= (A.seg[si++].rows + UM_M - 1) / UM_M;
        Tl.si = si;
        Tl.m0 = A.seg[si].row0 + mt * UM_M;
        Tl.m_end = A.seg[si].row0 + A.seg[si].rows;
      }
      fn(Tl);
    }
  };
  auto wait = [&](uint64_t* b, uint32_t parity) -> bool {
    if (!ok) return false;
    if (!mbar_wait_sleep(smem_u32(b), parity, A.wait_sleep_ns)) {
      ok = false;
      atomicOr(A.status, STATUS_TIMEOUT);
    }
    return ok;
  };

  if (warp >= 1 && warp <= 3) {
    // ---------------- producers ----------------
    // Every producer thread arrives on full[s] through its cp.async copies
    // (the arrival fires when they land), and thread 0 also arrives with the
    // transaction bytes of the slot's tensor copies: no producer waits for its
    // own copies, so the ring runs S chunks ahead of the MMAs.
    const int pt = tid - 32;   // 0..95
    uint32_t c = 0;
    if (tma && pt == 0) {
      // the encoded maps only: dense [2 * seg + part]; int4 codes [0], scale/bias [2]
      // (and the gate's [1], [3])
      auto prefetch = [&](int i) {
        asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&A.tm[i])) : "memory");
      };
      if (A.a_mode == UA_DENSE) {
        for (int si = 0; si < A.nseg; ++si)
          for (int p = 0; p < A.seg[si].nparts; ++p) prefetch(2 * si + p);
      } else {
        prefetch(0);
        prefetch(2);
        if (gated) { prefetch(1); prefetch(3); }
      }
    }
    if (A.tma_b && pt == 0) {
      asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&A.tm[8])) : "memory");
    }
    if (all_tma && pt != 0) ok = false;   // nothing to copy for the other producers (local flag only)
    tiles([&](const UmmaTile& Tl) {
      const int m0 = Tl.m0, n0 = Tl.n0, nvalid = Tl.nvalid;
      const UmmaGroup& G = Tl.G;
      // source rows of this thread's B pieces (i = pt + 96 q): fixed for the
      // tile, looked up once (a dependent global load per chunk otherwise)
      int brow[UM_BPIECES];
#pragma unroll
      for (int q = 0; q < UM_BPIECES; ++q) {
        const int n = (pt + 96 * q) >> 3;
        brow[q] = -1;
        if (n < nvalid && !A.tma_b) {
          if (A.experts && A.b_sorted) {
            brow[q] = G.p0 + n0 + n;
          } else if (A.experts) {
            const int pid = umma_pair(A, G.p0 + n0 + n);
            brow[q] = A.by_pair ? pid : pid / A.k;
          } else {
            brow[q] = n0 + n;
          }
        }
      }
      // slot i holds chunks SUB * i .. (a tile's last slot may hold fewer: the
      // copies past K read as zeros and no MMA reads them)
      for (int it = 0; ok && it < Tl.nit; it += SUB) {
        const int s = c % S;
        if (pt == 0) stamp(c, 0);
        if (c >= static_cast<uint32_t>(S) && !wait(&empty[s], ((c / S) - 1) & 1)) return;
        if (pt == 0) stamp(c, 1);
        char* slot = base + static_cast<size_t>(s) * P.stage;
        const uint32_t sa = smem_u32(slot), sbb = smem_u32(slot + P.a_raw);
        const uint32_t fb = smem_u32(&full[s]);
        const int k0 = (Tl.kc_begin + it) * UM_KC;
        if ((tma || A.tma_b) && pt == 0) {
          // the slot's tensor copies, all counted on full[s].  Every innermost
          // coordinate is a multiple of 16 bytes: dense A and B columns are
          // multiples of 64 elements (128 bytes), code words k0 / 8 are
          // multiples of 8 words (32 bytes), scale/bias rows m0 multiples of
          // 128 words; destinations are 1024-byte (swizzled tiles) or 128-byte
          // aligned (codes, scale/bias), as the plan guarantees.

          uint32_t tx = 0;
          if (tma) tx += A.a_mode == UA_DENSE ? static_cast<uint32_t>(UM_A_BYTES)
                                              : (gated ? 2u : 1u) * (CB + P.sb_box);
          if (A.tma_b) tx += P.b_bytes;
          mbar_arrive_expect_tx(fb, tx);
          stamp(c, 2);
          if (tma && A.a_mode == UA_DENSE) {
            // the tile's 128 rows x 64 columns of its segment (rows past the
            // segment's end read as zeros)
            const DenseSeg& Sg = A.seg[Tl.si];
            const int p = (Sg.nparts > 1 && k0 >= Sg.part[1].k0) ? 1 : 0;
            tma_load_2d(sa, &A.tm[2 * Tl.si + p], k0 - Sg.part[p].k0, m0 - Sg.row0, fb);
            stamp(c, 3);
          } else if (tma) {
            // codes (128 rows x 32 bytes) and the chunk's scale/bias words
            tma_load_3d(sa, &A.tm[0], k0 >> 3, m0, G.e, fb);
            stamp(c, 3);
            tma_load_3d(sa + CB, &A.tm[2], m0, k0 / A.G, G.e, fb);
            if (gated) {
              tma_load_3d(sa + CB + SBB, &A.tm[1], k0 >> 3, m0, G.e, fb);
              tma_load_3d(sa + 2 * CB + SBB, &A.tm[3], m0, k0 / A.G, G.e, fb);
            }
          }
          // B rows n0.. of the tile (dense tokens, or the pairs' sorted hidden
          // rows), one 64-column tile per chunk of the slot
          if (A.tma_b)
            for (int j = 0; j < SUB; ++j)
              tma_load_2d(sbb + j * P.b_tile, &A.tm[8], k0 + j * UM_KC, A.experts ? G.p0 + n0 : n0, fb);
          stamp(c, 4);
        }
        if (!tma && A.a_mode == UA_DENSE) {
          const DenseSeg& Sg = A.seg[Tl.si];
          for (int i = pt; i < UM_M * 8; i += 96) {
            const int r = i >> 3, j = i & 7;
            const int m = m0 + r, kk = k0 + 8 * j;
            const void* src = A.b0;
            uint32_t nbytes = 0;
            if (m < Tl.m_end) {
              for (int p = 0; p < Sg.nparts; ++p) {
                const DensePart& Pt = Sg.part[p];
                if (kk >= Pt.k0 && kk < Pt.k0 + Pt.wk) {
                  src = static_cast<const char*>(Pt.w) +
                        (static_cast<int64_t>(m - Sg.row0) * Pt.wk + (kk - Pt.k0)) * 2;
                  nbytes = 16;
                }
              }
            }
            cp_async16(sa + sw_off(r, 8 * j), src, nbytes);
          }
        } else if (!tma) {
          // codes: row r, 32 codes (16 bytes) per half
          for (int i = pt; i < UM_M * 2; i += 96) {
            const int r = i >> 1, hh = i & 1;
            const int m = min(m0 + r, A.n_rows - 1);
            const int64_t row = static_cast<int64_t>(G.e) * A.n_rows + m;
            const uint32_t nb = (m0 + r < A.n_rows) ? 16u : 0u;
            cp_async16(sa + r * 32 + hh * 16, A.q + row * (A.K >> 3) + (k0 >> 3) + 4 * hh, nb);
            if (gated)
              cp_async16(sa + CB + SBB + r * 32 + hh * 16,
                         A.q2 + row * (A.K >> 3) + (k0 >> 3) + 4 * hh, nb);
          }
        }
        if (A.a_mode == UA_INT4 && !tma) {
          // scale/bias words, group-major in the slot ([group of the chunk][row]):
          // one word per row (G >= 64), two (G = 32)
          for (int r = pt; r < UM_M; r += 96) {
            const int m = min(m0 + r, A.n_rows - 1);
            const int64_t row = static_cast<int64_t>(G.e) * A.n_rows + m;
            const int gw = k0 / A.G;
            for (int h2 = 0; h2 < (A.G == 32 ? 2 : 1); ++h2) {
              cp_async4(sa + CB + (h2 * 128 + r) * 4, A.sb + row * ngr + gw + h2);
              if (gated)
                cp_async4(sa + 2 * CB + SBB + (h2 * 128 + r) * 4, A.sb2 + row * ngr + gw + h2);
            }
          }
        }
        // B: the tile's valid tokens x 8 pieces of 16 bytes (padding rows only
        // reach accumulator columns that are never read: left as they are)
#pragma unroll
        for (int q = 0; q < UM_BPIECES; ++q) {
          if (brow[q] >= 0 && !A.tma_b) {
            const int i = pt + 96 * q;
            const int n = i >> 3, j = i & 7;
            cp_async16(sbb + sw_off(n, 8 * j),
                       static_cast<const char*>(A.b0) +
                           (A.b0_off + static_cast<int64_t>(brow[q]) * A.b0_stride + k0 + 8 * j) * 2,
                       16u);
          }
        }
        // pieces past the table (tiles wider than 128 tokens: dense only)
        for (int i = pt + 96 * UM_BPIECES; !A.tma_b && i < nvalid * 8; i += 96) {
          const int n = i >> 3, j = i & 7;
          int row = n0 + n;
          if (A.experts && A.b_sorted) {
            row = G.p0 + n0 + n;
          } else if (A.experts) {
            const int pid = umma_pair(A, G.p0 + n0 + n);
            row = A.by_pair ? pid : pid / A.k;
          }
          cp_async16(sbb + sw_off(n, 8 * j),
                     static_cast<const char*>(A.b0) + (A.b0_off + static_cast<int64_t>(row) * A.b0_stride + k0 + 8 * j) * 2,
                     16u);
        }
        if (pt == 0) stamp(c, 11);
        if (!all_tma) cp_async_mbar_arrive(fb);
        if (pt == 0) stamp(c, 10);
        ++c;
      }
    });
    cp_async_wait(0);
    // tensor copies still in flight land before the CTA ends: the last use of
    // each slot (already complete unless a wait gave up; bounded)
    if ((tma || A.tma_b) && pt == 0 && !ok)
      for (uint32_t j = c > static_cast<uint32_t>(S) ? c - S : 0u; j < c; ++j)
        mbar_wait(smem_u32(&full[j % S]), (j / S) & 1);
  } else if (warp >= 4) {
    // ---------------- dequant and epilogue ----------------
    const int dt = tid - 128;   // 0..127: row of the A tile
    uint32_t c = 0, q = 0, t = 0;   // chunks, ring slots, tiles
    tiles([&](const UmmaTile& Tl) {
      const int n0 = Tl.n0, nvalid = Tl.nvalid, npad = Tl.npad;
      const UmmaGroup& G = Tl.G;
      for (int it = 0; ok && it < Tl.nit; ++it) {
        const int j = it % SUB;   // chunk within the slot
        const int s = q % S, b = c % NA;
        if (j == 0 && !wait(&full[s], (q / S) & 1)) return;
        if (dt == 0) stamp(c, 5);
        if (c >= static_cast<uint32_t>(NA) && !wait(&dempty[b], ((c / NA) - 1) & 1)) return;
        if (dt == 0) stamp(c, 6);
        if (A.a_mode == UA_INT4) {
          const char* slot = base + static_cast<size_t>(s) * P.stage;
          const int r = dt;
          for (int gsel = 0; gsel < (gated ? 2 : 1); ++gsel) {
            const char* raw = slot + gsel * (CB + SBB);
            char* dst = base + P.abuf + static_cast<size_t>(b + NA * gsel) * UM_A_BYTES;
#pragma unroll
            for (int hh = 0; hh < 2; ++hh) {
              // codes: row r's 32 * SUB bytes; scale/bias: the slot's groups x 128 rows
              const uint4 w = *reinterpret_cast<const uint4*>(raw + r * (32 * SUB) + 32 * j + hh * 16);
              const int grp = (UM_KC * j + 32 * hh) / A.G;
              const uint32_t sbw = *reinterpret_cast<const uint32_t*>(raw + CB + (grp * 128 + r) * 4);
              const uint32_t ws[4] = {w.x, w.y, w.z, w.w};
              if (A.s_dt == A.mma_dt) {
                // packed 16-bit affine (scale and bias already in the MMA type)
                const uint32_t s2 = __byte_perm(sbw, 0u, 0x1010), b2 = __byte_perm(sbw, 0u, 0x3232);
#pragma unroll
                for (int i = 0; i < 4; ++i) {
                  uint32_t pr[4];
                  dq8_packed(ws[i], s2, b2, A.mma_dt, pr);
                  *reinterpret_cast<uint4*>(dst + sw_off(r, 32 * hh + 8 * i)) = make_uint4(pr[0], pr[1], pr[2], pr[3]);
                }
              } else {
                float sc, bi;
                sb_decode(sbw, A.s_dt, sc, bi);
#pragma unroll
                for (int i = 0; i < 4; ++i) {
                  uint32_t pr[4];
#pragma unroll
                  for (int j = 0; j < 4; ++j) {
                    const float lo = fmaf(sc, code_f((ws[i] >> (8 * j)) & 0xFu), bi);
                    const float hi = fmaf(sc, code_f((ws[i] >> (8 * j + 4)) & 0xFu), bi);
                    pr[j] = pack16(lo, hi, A.mma_dt);
                  }
                  *reinterpret_cast<uint4*>(dst + sw_off(r, 32 * hh + 8 * i)) = make_uint4(pr[0], pr[1], pr[2], pr[3]);
                }
              }
            }
          }
        }
        fence_proxy_async();
        mbar_arrive(smem_u32(&dfull[b]));
        if (dt == 0) stamp(c, 7);
        ++c;
        if (j == SUB - 1 || it == Tl.nit - 1) ++q;
      }
      // the tile's accumulators -> epilogue (rows 32 * (warp % 4) + lane)
      if (!wait(accb, t & 1)) return;
      tc_fence_after();
      const int q4 = warp & 3;
      const int m = Tl.m0 + 32 * q4 + lane;
      for (int c0 = 0; c0 < npad; c0 += 16) {
        float acc[16], accg[16];
        tmem_ld16(tmem + (static_cast<uint32_t>(32 * q4) << 16) + c0, acc);
        if (gated) tmem_ld16(tmem + (static_cast<uint32_t>(32 * q4) << 16) + 256 + c0, accg);
        if (m >= Tl.m_end) continue;
#pragma unroll
        for (int i = 0; i < 16; ++i) {
          const int n = c0 + i;
          if (n >= nvalid) break;
          const int pid = A.experts ? umma_pair(A, G.p0 + n0 + n) : n0 + n;
          if (A.ksplit > 1)
            A.part[(static_cast<int64_t>(Tl.split) * A.n_tokens + pid) * A.n_rows + m] = acc[i];
          else
            umma_epilogue(A, pid, m, acc[i], gated ? accg[i] : 0.f, gated,
                          A.out_sorted ? G.p0 + n0 + n : pid);
        }
      }
      tc_fence_before();
      mbar_arrive(smem_u32(epib));
      ++t;
    });
  } else if (lane == 0) {
    // ---------------- MMA issuer (warp 0, lane 0) ----------------
    uint32_t c = 0, q = 0, t = 0;   // chunks, ring slots, tiles
    tiles([&](const UmmaTile& Tl) {
      const int nit = Tl.nit;
      if (t > 0 && !wait(epib, (t - 1) & 1)) return;   // the previous tile's accumulators were read
      tc_fence_after();
      const uint32_t idesc = umma_idesc(Tl.npad, A.mma_dt);
      for (int it = 0; ok && it < nit; ++it) {
        const int j = it % SUB;
        const int s = q % S, b = c % NA;
        if (!wait(&dfull[b], (c / NA) & 1)) return;
        stamp(c, 8);
        fence_proxy_async();
        tc_fence_after();
        const char* slot = base + static_cast<size_t>(s) * P.stage;
        const uint32_t a_addr = A.a_mode == UA_DENSE ? smem_u32(slot)
                                                     : smem_u32(base + P.abuf + static_cast<size_t>(b) * UM_A_BYTES);
        const uint32_t b_addr = smem_u32(slot + P.a_raw + j * P.b_tile);
#pragma unroll
        for (int kk = 0; kk < UM_KC / 16; ++kk) {
          const uint64_t ad = umma_desc_sw128(a_addr + kk * 32);
          const uint64_t bd = umma_desc_sw128(b_addr + kk * 32);
          umma_f16(tmem, ad, bd, idesc, (it | kk) ? 1u : 0u);
          if (gated) {
            const uint32_t a2 = smem_u32(base + P.abuf + static_cast<size_t>(b + NA) * UM_A_BYTES);
            umma_f16(tmem + 256, umma_desc_sw128(a2 + kk * 32), bd, idesc, (it | kk) ? 1u : 0u);
          }
        }
        if (j == SUB - 1 || it == nit - 1) {   // the slot's last chunk: it may be refilled
          umma_commit(smem_u32(&empty[s]));
          ++q;
        }
        umma_commit(smem_u32(&dempty[b]));
        if (it == nit - 1) umma_commit(smem_u32(accb));
        stamp(c, 9);
        ++c;
      }
      ++t;
    });
    // every MMA issued has completed before tensor memory is released (a
    // commit tracks all earlier MMAs of this thread; bounded wait)
    umma_commit(smem_u32(drainb));
    mbar_wait(smem_u32(drainb), 0);
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 0) {
    tc_fence_after();
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(ncols));
  }
}

}  // namespace moe
