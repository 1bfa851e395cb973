// Row-grouped GEMM on tcgen05 with warp-specialised roles (k_umma2).
//
// Same contraction, operands, shared-memory layouts and epilogue as k_umma
// (moe_umma.cuh), but the three jobs of a K-chunk run in different warps and
// meet on mbarriers instead of CTA barriers, so copies, int4 dequantisation
// and tensor-core MMAs of different chunks overlap:
//
//   warps 1-3  producers: cp.async of the A operand (int4 codes and their
//              scale/bias words, or 16-bit rows) and of the B operand (the
//              tokens' 16-bit rows) of chunk c into ring slot c % S.  They
//              arrive on full[s] once their copies of the chunk have landed
//              (cp.async groups, S - 2 chunks in flight per thread).
//   warps 4-7  dequant: int4 -> 16-bit A tile in buffer c & 1 (after full[s]
//              and after the MMAs of chunk c - 2 released the buffer), then
//              arrive on dfull[c & 1].  After a tile's last chunk they read
//              the accumulators from tensor memory and write the epilogue.
//   warp 0     lane 0 issues the tcgen05.mma of chunk c once dfull[c & 1]
//              completes and commits them to empty[c % S] (the slot may be
//              refilled), dempty[c & 1] (the A buffer may be rewritten) and,
//              after a tile's last chunk, acc (the accumulators are final).
//
// Every role walks the same sequence of tiles and chunks, so the barrier
// phases are implied by the chunk and tile counts.  Every wait is bounded;
// on a timeout the role sets the status word's timeout bit and stops, the
// other roles' waits then run out too, and the kernel drains its copies and
// MMAs (bounded) before it frees tensor memory.
#pragma once

#include "moe_umma.cuh"

namespace moe {

__device__ __forceinline__ void mbar_arrive(uint32_t mbar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(mbar) : "memory");
}

__global__ void __launch_bounds__(UM_THREADS, 2) k_umma2(const __grid_constant__ UmmaArgs A) {
  extern __shared__ __align__(1024) char um_smem[];
  const bool gated = (A.a_mode == UA_INT4) && A.q2 != nullptr;
  const UmmaPlan P = umma_plan(A.a_mode, gated, A.n_tile, A.stages);
  char* base = um_smem;
  const int S = A.stages;
  // barriers and the tensor-memory address in the plan's token-table area
  uint64_t* bars = reinterpret_cast<uint64_t*>(base + P.tok);
  uint64_t* full = bars;               // [S]  producers' copies landed (96 arrivals)
  uint64_t* empty = bars + S;          // [S]  MMAs of the slot's chunk done (commit)
  uint64_t* dfull = bars + 2 * S;      // [2]  A tile ready (128 arrivals)
  uint64_t* dempty = dfull + 2;        // [2]  MMAs reading the A tile done (commit)
  uint64_t* accb = dempty + 2;         // [1]  a tile's accumulators final (commit)
  uint64_t* epib = accb + 1;           // [1]  the epilogue has read them (128 arrivals)
  uint64_t* drainb = epib + 1;         // [1]  every MMA issued has completed (final commit)
  uint32_t* tmem_holder = reinterpret_cast<uint32_t*>(drainb + 1);
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int ncols = gated ? 512 : 256;

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
      mbar_init(smem_u32(&full[s]), 96);
      mbar_init(smem_u32(&empty[s]), 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(smem_u32(&dfull[b]), 128);
      mbar_init(smem_u32(&dempty[b]), 1);
    }
    mbar_init(smem_u32(accb), 1);
    mbar_init(smem_u32(epib), 128);
    mbar_init(smem_u32(drainb), 1);
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_holder;

  const int n_groups = A.experts ? A.meta[0] : 1;
  const int mtiles = (A.n_rows + UM_M - 1) / UM_M;
  const int nkc = A.K / UM_KC;
  const int ngr = A.K / A.G;
  const int nsplit = A.ksplit > 1 ? A.ksplit : 1;
  const int nunits = n_groups * mtiles * nsplit;
  bool ok = true;

  // Walk the tiles of this CTA: fn(split, m0, kc_begin, nit, G, n0, nvalid, npad)
  auto tiles = [&](auto&& fn) {
    for (int unit = blockIdx.x; ok && unit < nunits; unit += gridDim.x) {
      const int split = unit % nsplit;
      const int gm = unit / nsplit;
      const int g = gm / mtiles, mt = gm - g * mtiles;
      const int kc_begin = static_cast<int>(static_cast<int64_t>(split) * nkc / nsplit);
      const int nit = static_cast<int>(static_cast<int64_t>(split + 1) * nkc / nsplit) - kc_begin;
      const UmmaGroup G = umma_group(A, g);
      for (int n0 = 0; ok && n0 < G.n; n0 += A.n_tile) {
        const int nvalid = min(A.n_tile, G.n - n0);
        fn(split, mt * UM_M, kc_begin, nit, G, n0, nvalid, (nvalid + 15) & ~15);
      }
    }
  };
  auto wait = [&](uint64_t* b, uint32_t parity) -> bool {
    if (!ok) return false;
    if (!mbar_wait(smem_u32(b), parity)) {
      ok = false;
      atomicOr(A.status, STATUS_TIMEOUT);
    }
    return ok;
  };

  if (warp >= 1 && warp <= 3) {
    // ---------------- producers ----------------
    const int pt = tid - 32;   // 0..95
    uint32_t c = 0, arrived = 0;
    auto arrive_landed = [&](int keep) {
      // chunks issued but not yet announced: all but `keep` of them have landed
      while (c - arrived > static_cast<uint32_t>(keep)) {
        const int n_pending = static_cast<int>(c - arrived) - 1;
        cp_async_wait(n_pending < 0 ? 0 : n_pending);
        fence_proxy_async();
        mbar_arrive(smem_u32(&full[arrived % S]));
        ++arrived;
      }
    };
    tiles([&](int, int m0, int kc_begin, int nit, const UmmaGroup& G, int n0, int nvalid, int npad) {
      for (int it = 0; ok && it < nit; ++it) {
        const int s = c % S;
        if (c >= static_cast<uint32_t>(S) && !wait(&empty[s], ((c / S) - 1) & 1)) return;
        char* slot = base + static_cast<size_t>(s) * P.stage;
        const uint32_t sa = smem_u32(slot), sbb = smem_u32(slot + P.a_raw);
        const int k0 = (kc_begin + it) * UM_KC;
        if (A.a_mode == UA_DENSE) {
          for (int i = pt; i < UM_M * 8; i += 96) {
            const int r = i >> 3, j = i & 7;
            const int m = m0 + r, kk = k0 + 8 * j;
            const void* src = A.b0;
            uint32_t nbytes = 0;
            if (m < A.n_rows) {
              int si = 0;
              while (m >= A.seg[si].row0 + A.seg[si].rows) ++si;
              const DenseSeg& Sg = A.seg[si];
              for (int p = 0; p < Sg.nparts; ++p) {
                const DensePart& Pt = Sg.part[p];
                if (kk >= Pt.k0 && kk < Pt.k0 + Pt.wk) {
                  src = static_cast<const char*>(Pt.w) +
                        (static_cast<int64_t>(m - Sg.row0) * Pt.wk + (kk - Pt.k0)) * 2;
                  nbytes = 16;
                }
              }
            }
            cp_async16(sa + core_off(r, 8 * j), src, nbytes);
          }
        } else {
          // codes: row r, 32 codes (16 bytes) per half
          for (int i = pt; i < UM_M * 2; i += 96) {
            const int r = i >> 1, hh = i & 1;
            const int m = min(m0 + r, A.n_rows - 1);
            const int64_t row = static_cast<int64_t>(G.e) * A.n_rows + m;
            const uint32_t nb = (m0 + r < A.n_rows) ? 16u : 0u;
            cp_async16(sa + r * 32 + hh * 16, A.q + row * (A.K >> 3) + (k0 >> 3) + 4 * hh, nb);
            if (gated)
              cp_async16(sa + UM_CODE_BYTES + UM_SB_BYTES + r * 32 + hh * 16,
                         A.q2 + row * (A.K >> 3) + (k0 >> 3) + 4 * hh, nb);
          }
          // scale/bias words: one word per row (G >= 64), two (G = 32)
          for (int r = pt; r < UM_M; r += 96) {
            const int m = min(m0 + r, A.n_rows - 1);
            const int64_t row = static_cast<int64_t>(G.e) * A.n_rows + m;
            const int gw = k0 / A.G;
            if (A.G == 32) {
              cp_async8(sa + UM_CODE_BYTES + r * 8, A.sb + row * ngr + gw);
              if (gated) cp_async8(sa + 2 * UM_CODE_BYTES + UM_SB_BYTES + r * 8, A.sb2 + row * ngr + gw);
            } else {
              cp_async4(sa + UM_CODE_BYTES + r * 8, A.sb + row * ngr + gw);
              if (gated) cp_async4(sa + 2 * UM_CODE_BYTES + UM_SB_BYTES + r * 8, A.sb2 + row * ngr + gw);
            }
          }
        }
        // B: npad tokens x 8 chunks of 16 bytes
        for (int i = pt; i < npad * 8; i += 96) {
          const int n = i >> 3, j = i & 7;
          const void* src = A.b0;
          uint32_t nbytes = 0;
          if (n < nvalid) {
            int row = n0 + n;
            if (A.experts) {
              const int pid = A.meta[2 + 2 * A.umax + G.p0 + n0 + n];
              row = A.by_pair ? pid : pid / A.k;
            }
            src = static_cast<const char*>(A.b0) + (A.b0_off + static_cast<int64_t>(row) * A.b0_stride + k0 + 8 * j) * 2;
            nbytes = 16;
          }
          cp_async16(sbb + core_off(n, 8 * j), src, nbytes);
        }
        cp_async_commit();
        ++c;
        arrive_landed(S - 2);
      }
    });
    cp_async_wait(0);
    arrive_landed(0);
  } else if (warp >= 4) {
    // ---------------- dequant and epilogue ----------------
    const int dt = tid - 128;   // 0..127: row of the A tile
    uint32_t c = 0, t = 0;
    tiles([&](int split, int m0, int, int nit, const UmmaGroup& G, int n0, int nvalid, int npad) {
      for (int it = 0; ok && it < nit; ++it) {
        const int s = c % S, b = c & 1;
        if (!wait(&full[s], (c / S) & 1)) return;
        if (c >= 2 && !wait(&dempty[b], ((c >> 1) - 1) & 1)) return;
        if (A.a_mode == UA_INT4) {
          const char* slot = base + static_cast<size_t>(s) * P.stage;
          const int r = dt;
          for (int gsel = 0; gsel < (gated ? 2 : 1); ++gsel) {
            const char* raw = slot + gsel * (UM_CODE_BYTES + UM_SB_BYTES);
            char* dst = base + P.abuf + static_cast<size_t>(b + 2 * gsel) * UM_A_BYTES;
#pragma unroll
            for (int hh = 0; hh < 2; ++hh) {
              const uint4 w = *reinterpret_cast<const uint4*>(raw + r * 32 + hh * 16);
              const uint32_t sbw = *reinterpret_cast<const uint32_t*>(
                  raw + UM_CODE_BYTES + r * 8 + ((A.G == 32) ? 4 * hh : 0));
              float sc, bi;
              sb_decode(sbw, A.s_dt, sc, bi);
              const uint32_t ws[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
              for (int i = 0; i < 4; ++i) {
                uint32_t pr[4];
#pragma unroll
                for (int j = 0; j < 4; ++j) {
                  const float lo = fmaf(sc, code_f((ws[i] >> (8 * j)) & 0xFu), bi);
                  const float hi = fmaf(sc, code_f((ws[i] >> (8 * j + 4)) & 0xFu), bi);
                  pr[j] = pack16(lo, hi, A.mma_dt);
                }
                *reinterpret_cast<uint4*>(dst + core_off(r, 32 * hh + 8 * i)) = make_uint4(pr[0], pr[1], pr[2], pr[3]);
              }
            }
          }
        }
        fence_proxy_async();
        mbar_arrive(smem_u32(&dfull[b]));
        ++c;
      }
      // the tile's accumulators -> epilogue (rows 32 * (warp % 4) + lane)
      if (!wait(accb, t & 1)) return;
      tc_fence_after();
      const int q4 = warp & 3;
      const int m = m0 + 32 * q4 + lane;
      for (int c0 = 0; c0 < npad; c0 += 16) {
        float acc[16], accg[16];
        tmem_ld16(tmem + (static_cast<uint32_t>(32 * q4) << 16) + c0, acc);
        if (gated) tmem_ld16(tmem + (static_cast<uint32_t>(32 * q4) << 16) + 256 + c0, accg);
        if (m >= A.n_rows) continue;
#pragma unroll
        for (int i = 0; i < 16; ++i) {
          const int n = c0 + i;
          if (n >= nvalid) break;
          const int pid = A.experts ? A.meta[2 + 2 * A.umax + G.p0 + n0 + n] : n0 + n;
          if (A.ksplit > 1)
            A.part[(static_cast<int64_t>(split) * A.n_tokens + pid) * A.n_rows + m] = acc[i];
          else
            umma_epilogue(A, pid, m, acc[i], gated ? accg[i] : 0.f, gated);
        }
      }
      tc_fence_before();
      mbar_arrive(smem_u32(epib));
      ++t;
    });
  } else if (lane == 0) {
    // ---------------- MMA issuer (warp 0, lane 0) ----------------
    uint32_t c = 0, t = 0;
    tiles([&](int, int, int, int nit, const UmmaGroup&, int, int, int npad) {
      if (t > 0 && !wait(epib, (t - 1) & 1)) return;   // the previous tile's accumulators were read
      tc_fence_after();
      const uint32_t idesc = umma_idesc(npad, A.mma_dt);
      for (int it = 0; ok && it < nit; ++it) {
        const int s = c % S, b = c & 1;
        if (!wait(&dfull[b], (c >> 1) & 1)) return;
        tc_fence_after();
        const char* slot = base + static_cast<size_t>(s) * P.stage;
        const uint32_t a_addr = A.a_mode == UA_DENSE ? smem_u32(slot)
                                                     : smem_u32(base + P.abuf + static_cast<size_t>(b) * UM_A_BYTES);
        const uint32_t b_addr = smem_u32(slot + P.a_raw);
#pragma unroll
        for (int kk = 0; kk < UM_KC / 16; ++kk) {
          const uint64_t ad = umma_desc(a_addr + kk * 2 * UM_LBO);
          const uint64_t bd = umma_desc(b_addr + kk * 2 * UM_LBO);
          umma_f16(tmem, ad, bd, idesc, (it | kk) ? 1u : 0u);
          if (gated) {
            const uint32_t a2 = smem_u32(base + P.abuf + static_cast<size_t>(b + 2) * UM_A_BYTES);
            umma_f16(tmem + 256, umma_desc(a2 + kk * 2 * UM_LBO), bd, idesc, (it | kk) ? 1u : 0u);
          }
        }
        umma_commit(smem_u32(&empty[s]));
        umma_commit(smem_u32(&dempty[b]));
        if (it == nit - 1) umma_commit(smem_u32(accb));
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
