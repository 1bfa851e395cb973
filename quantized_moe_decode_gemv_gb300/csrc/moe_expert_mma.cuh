// Expert projections of the gemv path on warp-level tensor-core MMAs (sm_103a).
//
// A routed expert's int4 matrix [n_rows, K] is contracted with the few token
// pairs routed to it.  Decoding every code to fp32 and multiplying on the CUDA
// cores costs several instructions per weight (the decode, one fma per pair),
// which keeps those kernels below the memory bandwidth as soon as a few pairs
// share an expert.  Here a warp computes a 16-row tile of the matrix for up to
// 4 * NTP pairs with mma.sync m16n8k16 (bf16 operands, fp32 accumulators):
//
//   * A holds 128 + q for the codes q (exact in bf16: the code fills the low
//     mantissa bits of 128.0).  The codes were re-laid at create time
//     (k_tile_codes) so that lane (g, t) of a warp reads, per 16-column block,
//     one word with exactly its eight codes: rows g and g + 8, columns t, t + 4,
//     t + 8, t + 12 of the block.  Three shifts and four masks-with-exponent
//     make its four bf16x2 fragment registers.
//   * Inside a block the MMA's k index runs through the permutation
//     (2t, 2t+1, 2t+8, 2t+9) -> (t, t+4, 8+t, 12+t); B is staged in the same
//     order, so the contraction is the plain sum over the block.
//   * B holds each pair's input row as two bf16 columns, hi = bf16(x) and
//     lo = bf16(x - hi): exact for 16-bit inputs, about 2^-17 relative for
//     fp32 ones.  One 8-column n-tile carries four pairs.
//   * The MMAs of a group of G columns accumulate in fresh registers, folded
//     in fp32 with the group's scale and bias and X, the group's sum of
//     hi + lo (the values the MMAs saw, so that the 128 offset cancels):
//       y += s * ((d_hi + d_lo) - 128 X) + b X
//     (products (128 + q) x_hi are exact in fp32; the offset costs about
//     four bits of the fp32 accumulator, far inside the tolerance).
//
// Each output element depends on its own pair's column only (the MMA's columns
// are independent and every fold runs in a fixed order), so a row gives the
// same bits whatever the batch.
//
// The same kernel reads NVFP4 and MXFP4 experts (E2M1 codes in the same
// fragment order; A holds 128 + 2v + 12, exact in bf16) and folds each scale
// block (16 or 32 columns) with its E4M3 or E8M0 scale.  The work of a launch
// is the routing's units (distinct expert and pass of its pairs, 16-row tile)
// spread over a grid sized before the routing is known.
//
// Weights stream through a private ring per warp: lane 0 issues the bulk copies
// of one (16-row tile, CK x 64 columns) chunk -- the codes and the chunk's
// scale/bias words (gate and up for SwiGLU), each one contiguous range -- that
// complete on the stage's mbarrier; the warp waits (bounded), computes and
// refills the stage with its next chunk.  The down projection issues its first
// copies before it waits for the up projection (its experts are final once the
// routing is).  A wait that runs out sets the timeout bit of the status word;
// the warp then stops issuing, lets its copies in flight land (bounded) and
// skips its remaining arithmetic.
#pragma once

#include <cuda_bf16.h>

#include "moe_kernels.cuh"
#include "moe_expert_bulk.cuh"   // eb_smem, eb_bulk, eb_wait

namespace moe {

constexpr int EM_WARPS = 8;
constexpr int EM_NT = EM_WARPS * 32;
constexpr int EM_MAX_NTP = 4;          // n-tiles (4 pairs each) per pass over the weights
constexpr int EM_MAX_PAIRS = 4 * EM_MAX_NTP;

// Shared-memory plan of one k_expert_mma launch (host and device agree).
//   [B fragments: pp/4 n-tiles x K/16 blocks x 32 lanes x 8 bytes]
//   [group sums of x: pp x K/gx floats, 128-aligned (gx: G; 16 NVFP4; 32 MXFP4)]
//   [K-split partials (ks > 1): 2 x EM_WARPS x 4 NTP x 32 floats]
//   [rings: EM_WARPS x ns stages of stage_bytes]  [mbarriers: EM_WARPS x ns]
// A stage holds, per matrix (gate first for SwiGLU, then up), ck x 512 bytes of
// codes, then per matrix ck x 128 bytes of scale/bias words (the most a chunk
// needs: two 64-byte groups per 64 columns at G = 32).
struct EmPlan {
  int ck, ns, pp, ks;
  int stage_bytes, b_bytes, xs_bytes, red_off, ring_off, bar_off;
  int smem;
};

// n-tiles of accumulators of a pass of pp pairs (the kernel's NTP)
__host__ __device__ inline int em_ntp(int pp) { return pp <= 4 ? 1 : (pp <= 8 ? 2 : 4); }

__host__ __device__ inline EmPlan em_plan(int K, int G, bool gated, int ck, int ns, int pp, int ks, int gx = 0) {
  if (gx <= 0) gx = G;
  EmPlan p;
  p.ck = ck;
  p.ns = ns;
  p.pp = pp;
  p.ks = ks;
  p.stage_bytes = (gated ? 2 : 1) * ck * (512 + 128);
  p.b_bytes = (pp / 4) * (K / 16) * 256;
  p.xs_bytes = (pp * (K / gx) * 4 + 127) & ~127;
  p.red_off = p.b_bytes + p.xs_bytes;
  p.ring_off = p.red_off + (ks > 1 ? 2 * EM_WARPS * 4 * em_ntp(pp) * 32 * 4 : 0);
  p.bar_off = p.ring_off + EM_WARPS * ns * p.stage_bytes;
  p.smem = p.bar_off + EM_WARPS * ns * 8;
  return p;
}

// D += A * B for one m16n8k16 tile (bf16 operands, fp32 accumulators)
__device__ __forceinline__ void mma_16816(float (&d)[4], const uint32_t (&a)[4], uint32_t b0, uint32_t b1) {
  asm("mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
      "{%0,%1,%2,%3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

// A lane's word of a 16-column block -> its four bf16x2 fragment registers
// holding 128 + q (nibble i of the word goes to register i % 4, half i / 4;
// the code fills the low mantissa bits of 128.0, exactly)
__device__ __forceinline__ void em_decode(uint32_t w, uint32_t (&a)[4]) {
  constexpr uint32_t M = 0x43004300u;   // bf16 128.0 in both halves
#pragma unroll
  for (int i = 0; i < 4; ++i) a[i] = ((w >> (4 * i)) & 0x000F000Fu) | M;
}

// NVFP4 codes (E2M1: sign, two exponent bits, one mantissa bit; magnitudes
// 0, 0.5, 1, 1.5, 2, 3, 4, 6) -> the same four registers, holding 128 + n with
// n = 2 v + 12 in 0..24 (exact in bf16; the fold removes the 140 offset).  Two
// byte permutes look n up for four codes: the positive table by the code
// nibble, the negative one by the nibble with its sign bit flipped; a nibble
// whose bit 3 is set selects in sign-replicate mode, which yields 0x00 from
// these tables (every entry is below 0x80), so exactly one lookup is nonzero.
__device__ __forceinline__ uint32_t em_prmt(uint32_t a, uint32_t b, uint32_t sel) {
  uint32_t d;
  asm("prmt.b32 %0, %1, %2, %3;" : "=r"(d) : "r"(a), "r"(b), "r"(sel));
  return d;
}
__device__ __forceinline__ void em_decode_fp4(uint32_t w, uint32_t (&a)[4]) {
  constexpr uint32_t TP0 = 0x0F0E0D0Cu, TP1 = 0x18141210u;   // 12 + 2v, v = 0 .. 1.5 | 2 .. 6
  constexpr uint32_t TN0 = 0x090A0B0Cu, TN1 = 0x00040608u;   // 12 - 2v
  const uint32_t x = w ^ 0x88888888u;
  const uint32_t p0 = em_prmt(TP0, TP1, w) | em_prmt(TN0, TN1, x);               // codes 0..3
  const uint32_t p1 = em_prmt(TP0, TP1, w >> 16) | em_prmt(TN0, TN1, x >> 16);   // codes 4..7
  // register i: n of code i (byte 0) and of code i + 4 (byte 2); bytes 1 and 3
  // replicate the clear top bit of a table byte (0x00), then take 0x43
  a[0] = em_prmt(p0, p1, 0xC480u) | 0x43004300u;
  a[1] = em_prmt(p0, p1, 0xD591u) | 0x43004300u;
  a[2] = em_prmt(p0, p1, 0xE6A2u) | 0x43004300u;
  a[3] = em_prmt(p0, p1, 0xF7B3u) | 0x43004300u;
}

// Four E4M3 block scales (byte j: block j of a 64-column chunk) -> floats
// times m (exact conversions: every E4M3 value is an fp16 value)
__device__ __forceinline__ void em_e4m3x4(uint32_t w, float m, float (&s)[4]) {
  uint32_t h01, h23;
  asm("{\n\t.reg .b16 lo, hi;\n\tmov.b32 {lo, hi}, %2;\n\t"
      "cvt.rn.f16x2.e4m3x2 %0, lo;\n\tcvt.rn.f16x2.e4m3x2 %1, hi;\n\t}"
      : "=r"(h01), "=r"(h23)
      : "r"(w));
  const float2 f01 = __half22float2(*reinterpret_cast<const __half2*>(&h01));
  const float2 f23 = __half22float2(*reinterpret_cast<const __half2*>(&h23));
  s[0] = f01.x * m;
  s[1] = f01.y * m;
  s[2] = f23.x * m;
  s[3] = f23.y * m;
}

// An E8M0 scale byte (2^(b - 127); 0xFF is NaN) times m (a power of two: exact)
__device__ __forceinline__ float em_e8m0(uint32_t b, float m) {
  const uint32_t bits = b == 0u ? 0x00400000u : (b == 255u ? 0x7FC00000u : (b << 23));
  return __uint_as_float(bits) * m;
}

__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
  const __nv_bfloat162 r = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<const uint32_t*>(&r);
}

// Sixteen consecutive elements x[base .. base + 15] of an input row as fp32
// (vector loads where the row offset allows them).
__device__ __forceinline__ void em_ld16(const void* p, int dt, int64_t base, bool vec, float (&v)[16]) {
  if (dt == DT_FP32) {
    const float* f = static_cast<const float*>(p) + base;
    if (vec) {
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        const float4 a = __ldcg(reinterpret_cast<const float4*>(f) + q);
        v[4 * q] = a.x; v[4 * q + 1] = a.y; v[4 * q + 2] = a.z; v[4 * q + 3] = a.w;
      }
    } else {
#pragma unroll
      for (int q = 0; q < 16; ++q) v[q] = __ldcg(f + q);
    }
  } else if (vec) {
    const uint4* h = reinterpret_cast<const uint4*>(static_cast<const uint16_t*>(p) + base);
#pragma unroll
    for (int q = 0; q < 2; ++q) {
      const uint4 a = __ldcg(h + q);
      const uint32_t w[4] = {a.x, a.y, a.z, a.w};
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        v[8 * q + 2 * j] = dt == DT_BF16 ? bf16lo(w[j]) : f16lo(w[j]);
        v[8 * q + 2 * j + 1] = dt == DT_BF16 ? bf16hi(w[j]) : f16hi(w[j]);
      }
    }
  } else {
#pragma unroll
    for (int q = 0; q < 16; ++q) v[q] = ld16(p, base + q, dt);
  }
}

// NTP: n-tiles of accumulators (pairs per pass = 4 NTP; up to two n-tiles
// keep the registers for two CTAs per SM).  GB: 16-column blocks per scale
// group (G / 16).  FMT 1: NVFP4 codes (GB = 4: a row's scale word of a
// 64-column chunk holds the chunk's four E4M3 block scales), folded per
// 16-column block:
//   y += (S / 2) ((d_hi + d_lo) - 140 X),   S = E4M3 scale x matrix scale
// FMT 2: MXFP4 codes (GB = 4; a row's 16-bit scale entry of a 64-column chunk
// holds its two E8M0 block scales), folded the same way per 32-column block
// with S = the E8M0 scale.
template <bool GATED, int NTP, int GB, int FMT = 0>
__global__ void __launch_bounds__(EM_NT, NTP <= 2 ? 2 : 1) k_expert_mma(const __grid_constant__ ExpertArgs A) {
  extern __shared__ __align__(128) unsigned char em_smem_raw[];
  constexpr bool FP4 = FMT != 0, MX = FMT == 2;
  static_assert(!FP4 || GB == 4, "fp4 scales are staged per 64-column chunk");
  constexpr int G = 16 * GB;
  constexpr int GX = FMT == 1 ? 16 : (MX ? 32 : G), GBX = GX / 16;   // columns of a sum of x
  constexpr int NM = GATED ? 2 : 1;
  const int K = A.K, nkc = K >> 6, nkb = K >> 4, ngr = K / G, ngx = K / GX;
  const EmPlan P = em_plan(K, G, GATED, A.ck, A.nst, A.pp, A.ks, GX);
  const int CK = P.ck, NS = P.ns;
  uint2* bfrag = reinterpret_cast<uint2*>(em_smem_raw);
  float* xs = reinterpret_cast<float*>(em_smem_raw + P.b_bytes);
  float* red = reinterpret_cast<float*>(em_smem_raw + P.red_off);
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int g = lane >> 2, t = lane & 3;
  unsigned char* ring = em_smem_raw + P.ring_off + warp * NS * P.stage_bytes;
  uint64_t* bars = reinterpret_cast<uint64_t*>(em_smem_raw + P.bar_off) + warp * NS;

  const int ntiles = A.n_rows >> 4;
  const int* uniq_e = A.meta + 1;
  const int* uniq_p0 = A.meta + 1 + A.umax;
  const int* pairs = A.meta + 2 + 2 * A.umax;
  const long long n_pairs = static_cast<long long>(A.T) * A.k;

  if (lane == 0) {
    for (int s = 0; s < NS; ++s)
      asm volatile("mbarrier.init.shared::cta.b64 [%0], 1;" ::"r"(eb_smem(bars + s)) : "memory");
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  __syncwarp();
  cta_stamp(A.trace, 0);
  if (!A.pre_wait_phase) griddep_wait();
  griddep_launch();
  if (!A.pre_wait_phase) cta_stamp(A.trace, 1);

  // ---- work: the units (segment, 16-row tile) of this routing, a segment
  // being a distinct expert u and a pass of up to pp of its pairs, spread
  // evenly over the grid.  With at least 4 CTAs a segment (m = grid / nseg),
  // CTA j of a segment's m takes its tiles [j ntiles / m, (j + 1) ntiles / m):
  // one segment a CTA, the same ranges in every segment.  Otherwise CTA c
  // takes the units [c U / grid, (c + 1) U / grid) in segment-major order (U =
  // nseg ntiles), which may span segments.  (The grid is sized before the
  // routing is known; spreading by the units the routing made keeps every CTA
  // busy whatever the load, and spreads the tiles' combines over the CTAs.)
  __shared__ int s_seg[6];   // nseg, slot and pass of a segment, this CTA's units [u0, u1)
  auto npass_of = [&](int u) -> int {
    const int n = uniq_p0[u + 1] - uniq_p0[u];
    if (n <= 0 || (A.max_pairs > 0 && n > A.max_pairs)) return 0;
    return (n + P.pp - 1) / P.pp;
  };
  const int nslots = A.meta[0], gsz = static_cast<int>(gridDim.x), cta = static_cast<int>(blockIdx.x);
  // warp 0: slot u and pass of segment sgi (the slots' pass counts scanned 32 at
  // a time; the counts were just read, so these reads hit L1)
  auto lookup = [&](int sgi) {
    int base = 0;
    for (int u0 = 0; u0 < nslots; u0 += 32) {
      const int u = u0 + lane;
      const int v = u < nslots ? npass_of(u) : 0;
      int incl = v;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const int y = __shfl_up_sync(0xffffffffu, incl, o);
        if (lane >= o) incl += y;
      }
      const int tot = __shfl_sync(0xffffffffu, incl, 31);
      const unsigned hit = __ballot_sync(0xffffffffu, sgi < base + incl && sgi >= base + incl - v);
      if (hit) {
        if (lane == __ffs(hit) - 1) { s_seg[1] = u; s_seg[2] = sgi - (base + incl - v); }
        break;
      }
      base += tot;
    }
  };
  if (warp == 0) {
    // the segment count, this CTA's first segment and its tile range
    int cnt = 0;
    if (A.one_pass) {
      // every slot has at most pp pairs: the segments are the slots.  Their
      // entries come to L1 while the count is read.
      if (lane * 32 < 2 * A.umax + 1)
        asm volatile("prefetch.global.L1 [%0];" ::"l"(uniq_e + lane * 32));
      cnt = nslots;
    } else {
      for (int u = lane; u < nslots; u += 32) cnt += npass_of(u);
#pragma unroll
      for (int o = 16; o >= 1; o >>= 1) cnt += __shfl_xor_sync(0xffffffffu, cnt, o);
    }
    const int ns_ = cnt;
    int64_t u0 = 0, u1 = 0;
    if (ns_ > 0) {
      const int m = gsz / ns_;
      if (m >= 4) {
        // (the CTAs past nseg m stay idle)
        const int mm = min(ntiles, m), sgc = cta / mm, j = cta - sgc * mm;
        if (sgc < ns_) {
          u0 = static_cast<int64_t>(sgc) * ntiles + j * ntiles / mm;
          u1 = static_cast<int64_t>(sgc) * ntiles + (j + 1) * ntiles / mm;
        }
      } else {
        const int64_t U = static_cast<int64_t>(ns_) * ntiles;
        u0 = cta * U / gsz;
        u1 = (cta + 1) * U / gsz;
      }
    }
    if (lane == 0) { s_seg[0] = ns_; s_seg[3] = static_cast<int>(u0); s_seg[4] = static_cast<int>(u1); }
  }
  __syncthreads();
  const int nseg = s_seg[0];
  const int cu0 = s_seg[3], cu1 = s_seg[4];
  int sg = cu0 / ntiles;
  int tb = 0, te = 0;   // this CTA's tiles of segment sg

  // The CTA's warps form EM_WARPS / KS tile slots of KS warps; warp ks of slot
  // sl takes the tiles tb + sl + nslot ti, and of each its part of K in
  // chunks of CK 64-column blocks.  The slot's partial sums meet in shared
  // memory at the end of a tile.  The issuing lane and the computing warp walk
  // the same sequence with incremental counters.
  const int KS = P.ks, nslot = EM_WARPS / KS, slot = warp / KS, ks = warp - slot * KS;
  // K part of warp ks, in 64-column blocks [kc_lo, kc_hi): whole groups, and a
  // function of K and KS alone (not of the ring's chunk size, which the batch
  // size picks), so that a row's partial sums do not depend on the batch
  const int unit = G > 64 ? G / 64 : 1, nu = nkc / unit;
  const int kc_lo = (ks * nu / KS) * unit, kc_hi = ((ks + 1) * nu / KS) * unit;
  const int nit = (kc_hi - kc_lo + CK - 1) / CK;   // items (chunks) a tile
  int my_tiles = 0;
  const uint32_t* qm[2] = {GATED ? A.qt_gate : A.qt, A.qt};
  const uint32_t* sm[2] = {GATED ? A.sbt_gate : A.sbt, A.sbt};
  int64_t e = 0;                        // the segment's expert
  int total = 0;                        // this warp's items of the segment
  int iss_ti = 0, iss_ch = 0, iss_s = 0, issued = 0, iss_seg = 0;   // lane 0's issue position
  auto issue_next = [&]() {
    const int64_t tile = e * ntiles + tb + slot + nslot * iss_ti;
    const int kc0 = kc_lo + iss_ch * CK, ckt = min(CK, kc_hi - kc0);
    const int g0 = (kc0 * 64) / G, ng = (ckt * 64) / G;
    const uint32_t bar = eb_smem(bars + iss_s);
    unsigned char* st = ring + iss_s * P.stage_bytes;
    // scale bytes of the chunks: 64 per chunk (16 rows x one word), MXFP4 32
    // (16 rows x one 16-bit entry)
    const uint32_t sbytes = MX ? ckt * 32u : ng * 64u;
    const uint32_t bytes = NM * (ckt * 512u + sbytes);
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(bytes) : "memory");
#pragma unroll
    for (int m = 0; m < NM; ++m) {
      eb_bulk(eb_smem(st + m * CK * 512), qm[m] + (tile * nkc + kc0) * 128, ckt * 512u, bar);
      const void* ssrc = MX ? static_cast<const void*>(reinterpret_cast<const unsigned char*>(sm[m]) +
                                                        (tile * nkc + kc0) * 32)
                            : static_cast<const void*>(sm[m] + (tile * ngr + g0) * 16);
      eb_bulk(eb_smem(st + NM * CK * 512 + m * CK * 128), ssrc, sbytes, bar);
    }
    ++issued;
    ++iss_seg;
    if (++iss_s == NS) iss_s = 0;
    if (++iss_ch == nit) { iss_ch = 0; ++iss_ti; }
  };
  // the pair ids of a pass (-1: failed its index check)
  __shared__ int s_pid[EM_MAX_PAIRS];
  int p0 = 0, npp = 0, nnt = 0;
  // Segment sg: its slot and pass (warp 0 scans the slots' pass counts), its
  // pairs; the first copies of this warp's items go out at once.
  auto prepare = [&](int sgi) {
    tb = max(cu0 - sgi * ntiles, 0);
    te = min(cu1 - sgi * ntiles, ntiles);
    my_tiles = (te - tb > slot) ? (te - tb - slot + nslot - 1) / nslot : 0;
    if (warp == 0) {
      if (!A.one_pass) lookup(sgi);
      else if (lane == 0) { s_seg[1] = sgi; s_seg[2] = 0; }
    }
    __syncthreads();
    const int u = s_seg[1], pass = s_seg[2];
    // a bad slot (index checks) copies nothing and writes nothing
    const bool e_ok = idx_ok(A.status, CK_EXPERT_E, uniq_e[u], A.n_experts) &&
                      range_ok(A.status, uniq_p0[u], uniq_p0[u + 1], n_pairs);
    e = e_ok ? uniq_e[u] : 0;
    p0 = uniq_p0[u] + pass * P.pp;
    npp = e_ok ? min(P.pp, uniq_p0[u + 1] - p0) : 0;
    nnt = (npp + 3) >> 2;
    total = npp > 0 ? my_tiles * nit : 0;
    iss_ti = 0;
    iss_ch = 0;
    iss_seg = 0;
    if (lane == 0)
      for (int n0 = 0; n0 < min(NS, total); ++n0) issue_next();
    if (threadIdx.x < npp) {
      const int pid = pairs[p0 + threadIdx.x];
      s_pid[threadIdx.x] = idx_ok(A.status, CK_EXPERT_PAIR, pid, n_pairs) ? pid : -1;
    }
  };

  // input rows may be read as vectors when every row start is 16-byte aligned
  const bool xvec = A.xin_dt == DT_FP32 ? ((A.xin_off | A.xin_stride) & 3) == 0
                                        : ((A.xin_off | A.xin_stride) & 7) == 0;
  bool ok = true;
  int gi = 0, gi_fail = 0, cs = 0;   // items consumed; the next one's stage
  uint32_t phase = 0;                // its mbarrier phase
  __shared__ int s_cflag[EM_NT];
  // the down projection's metadata is final at launch: its first segment
  // (copies and pair ids) is prepared before the wait
  bool waited = !A.pre_wait_phase;
  for (bool first = true; cu0 < cu1 && sg * ntiles < cu1; ++sg, first = false) {
    if (!first) __syncthreads();   // every warp is done with the previous segment's B and ids
    prepare(sg);
    if (!waited) {
      griddep_wait();
      cta_stamp(A.trace, 1);
      waited = true;
    }
    __syncthreads();
    // ---- stage B: pair pl -> n-tile pl / 4, columns 2 (pl % 4) (hi) and + 1 (lo).
    // Thread i takes block kb of pair pl (i = pl * nkb + kb): its 16 elements,
    // the four lanes' B words of the hi and lo columns, and the block's sum of
    // hi + lo; the GB threads of a group are consecutive lanes (nkb and the
    // stride are multiples of GB) and add their sums by a fixed butterfly.  The
    // loop runs in whole warps (its count rounded up to 32) for the shuffles.
    const int nblk = nnt * 4 * nkb;
    for (int i = threadIdx.x; i < ((nblk + 31) & ~31); i += EM_NT) {
      const int pl = i / nkb, kb = i - pl * nkb;
      float v[16];
#pragma unroll
      for (int q = 0; q < 16; ++q) v[q] = 0.f;
      if (i < nblk && pl < npp) {
        const int pid = max(s_pid[pl], 0);
        const int64_t row = A.xin_by_pair ? pid : (pid / A.k);
        em_ld16(A.xin, A.xin_dt, A.xin_off + row * A.xin_stride + 16 * kb, xvec, v);
      }
      float sx = 0.f;
      if (i < nblk) {
        const int nt = pl >> 2, c = 2 * (pl & 3);
        uint2* dst = bfrag + (static_cast<int64_t>(nt) * nkb + kb) * 32;
#pragma unroll
        for (int tt = 0; tt < 4; ++tt) {
          float hi[4], lo[4];
#pragma unroll
          for (int j = 0; j < 4; ++j) {
            const float xv = v[tt + 4 * j];   // columns tt, tt + 4, tt + 8, tt + 12
            hi[j] = __bfloat162float(__float2bfloat16_rn(xv));
            lo[j] = __bfloat162float(__float2bfloat16_rn(xv - hi[j]));
            v[tt + 4 * j] = hi[j] + lo[j];   // the value the MMAs see
          }
          dst[c * 4 + tt] = make_uint2(pack_bf16x2(hi[0], hi[1]), pack_bf16x2(hi[2], hi[3]));
          dst[(c + 1) * 4 + tt] = make_uint2(pack_bf16x2(lo[0], lo[1]), pack_bf16x2(lo[2], lo[3]));
        }
#pragma unroll
        for (int q = 0; q < 16; q += 4) sx += (v[q] + v[q + 1]) + (v[q + 2] + v[q + 3]);
      }
#pragma unroll
      for (int o = 1; o < GBX; o <<= 1) sx += __shfl_xor_sync(0xffffffffu, sx, o);
      if (i < nblk && (kb & (GBX - 1)) == 0) xs[pl * ngx + kb / GBX] = sx;
    }
    __syncthreads();
    if (first) cta_stamp(A.trace, 6);

    // ---- this warp's tiles
    const uint2* bl = bfrag + lane;   // + (nt * nkb + kb) * 32
    const float* xsl = xs + t * ngx;  // + nt * 4 * ngx + grp
    // NVFP4: the segment's matrix scales, halved (the fold's 2 v); MXFP4: 1/2
    const float gsu = FMT == 1 ? 0.5f * __ldg(A.gsc + e) : 0.5f;
    const float gsg = (FMT == 1 && GATED) ? 0.5f * __ldg(A.gsc_gate + e) : 0.5f;
    float y[NTP][2], yg[NTP][2], acc[NTP][4], accg[NTP][4];
    // (a segment whose slot failed its index check issued no copies: no tiles)
    const int seg_tiles = npp > 0 ? my_tiles : 0;
    for (int ti = 0; ti < seg_tiles; ++ti) {
     const int rt = tb + slot + nslot * ti;
#pragma unroll
     for (int nt = 0; nt < NTP; ++nt) y[nt][0] = y[nt][1] = yg[nt][0] = yg[nt][1] = 0.f;
     for (int ch = 0; ch < nit; ++ch, ++gi) {
      const int kc0 = kc_lo + ch * CK, ckt = min(CK, kc_hi - kc0);
      const int g0 = (kc0 * 64) / G;
      if (ok && !eb_wait(eb_smem(bars + cs), phase)) {
        ok = false;
        gi_fail = gi;
        if (lane == 0) atomicOr(A.status, STATUS_TIMEOUT);
      }
      if (gi == 0) cta_stamp(A.trace, 7);
      if (ok) {
        const unsigned char* st = ring + cs * P.stage_bytes;
        const uint4* cq = reinterpret_cast<const uint4*>(st + (NM - 1) * CK * 512) + lane;   // up codes
        const uint4* cg = reinterpret_cast<const uint4*>(st) + lane;                        // gate codes
        const uint32_t* sbu = reinterpret_cast<const uint32_t*>(st + NM * CK * 512 + (NM - 1) * CK * 128) + g;
        const uint32_t* sbg = reinterpret_cast<const uint32_t*>(st + NM * CK * 512) + g;
#pragma unroll 1
        for (int c = 0; c < ckt; ++c) {
          // the chunk's four blocks: 128 + q in A, the MMAs of a group chained
          // in fresh accumulators, then the fold
          //   y += s ((d_hi + d_lo) - 128 X) + b X,   X = sum of the group's x
          const uint4 wq = cq[c * 32];
          uint4 wg = make_uint4(0u, 0u, 0u, 0u);
          if (GATED) wg = cg[c * 32];
          const uint32_t wqs[4] = {wq.x, wq.y, wq.z, wq.w};
          const uint32_t wgs[4] = {wg.x, wg.y, wg.z, wg.w};
          const uint2* bk = bl + static_cast<int64_t>(kc0 + c) * 4 * 32;
          if constexpr (FP4) {
            // rows g and g + 8: the chunk's block scales (NVFP4: four E4M3, times
            // gs / 2; MXFP4: two E8M0, times 1/2)
            float su0[4], su1[4], sg0[4], sg1[4];
            constexpr int NB = MX ? 2 : 4;   // scale blocks of a chunk
            if constexpr (MX) {
              const uint16_t* s16u = reinterpret_cast<const uint16_t*>(sbu - g) + g;
              const uint16_t* s16g = reinterpret_cast<const uint16_t*>(sbg - g) + g;
              const uint32_t w0 = s16u[c * 16], w1 = s16u[c * 16 + 8];
              su0[0] = em_e8m0(w0 & 0xFFu, gsu); su0[1] = em_e8m0(w0 >> 8, gsu);
              su1[0] = em_e8m0(w1 & 0xFFu, gsu); su1[1] = em_e8m0(w1 >> 8, gsu);
              if (GATED) {
                const uint32_t v0 = s16g[c * 16], v1 = s16g[c * 16 + 8];
                sg0[0] = em_e8m0(v0 & 0xFFu, gsg); sg0[1] = em_e8m0(v0 >> 8, gsg);
                sg1[0] = em_e8m0(v1 & 0xFFu, gsg); sg1[1] = em_e8m0(v1 >> 8, gsg);
              }
            } else {
              em_e4m3x4(sbu[c * 16], gsu, su0);
              em_e4m3x4(sbu[c * 16 + 8], gsu, su1);
              if (GATED) {
                em_e4m3x4(sbg[c * 16], gsg, sg0);
                em_e4m3x4(sbg[c * 16 + 8], gsg, sg1);
              }
            }
#pragma unroll
            for (int j = 0; j < 4; ++j) {
              constexpr int JB = 4 / NB;   // 16-column blocks of a scale block
              if (j % JB == 0) {
#pragma unroll
                for (int nt = 0; nt < NTP; ++nt)
#pragma unroll
                  for (int r = 0; r < 4; ++r) acc[nt][r] = accg[nt][r] = 0.f;
              }
              uint32_t a[4], ag[4];
              em_decode_fp4(wqs[j], a);
              if (GATED) em_decode_fp4(wgs[j], ag);
              const int q = j / JB;   // this block's scale
#pragma unroll
              for (int nt = 0; nt < NTP; ++nt) {
                if (nt < nnt) {
                  const uint2 b = bk[(static_cast<int64_t>(nt) * nkb + j) * 32];
                  mma_16816(acc[nt], a, b.x, b.y);
                  if (GATED) mma_16816(accg[nt], ag, b.x, b.y);
                  if (j % JB == JB - 1) {
                    const float xv = xsl[nt * 4 * ngx + (kc0 + c) * NB + q];
                    y[nt][0] = fmaf(su0[q], fmaf(-140.f, xv, acc[nt][0] + acc[nt][1]), y[nt][0]);
                    y[nt][1] = fmaf(su1[q], fmaf(-140.f, xv, acc[nt][2] + acc[nt][3]), y[nt][1]);
                    if (GATED) {
                      yg[nt][0] = fmaf(sg0[q], fmaf(-140.f, xv, accg[nt][0] + accg[nt][1]), yg[nt][0]);
                      yg[nt][1] = fmaf(sg1[q], fmaf(-140.f, xv, accg[nt][2] + accg[nt][3]), yg[nt][1]);
                    }
                  }
                }
              }
            }
          } else {
#pragma unroll
          for (int j = 0; j < 4; ++j) {
            if (j % GB == 0 && (GB <= 4 || (c & 1) == 0)) {
#pragma unroll
              for (int nt = 0; nt < NTP; ++nt)
#pragma unroll
                for (int r = 0; r < 4; ++r) acc[nt][r] = accg[nt][r] = 0.f;
            }
            uint32_t a[4], ag[4];
            em_decode(wqs[j], a);
            if (GATED) em_decode(wgs[j], ag);
#pragma unroll
            for (int nt = 0; nt < NTP; ++nt) {
              if (nt < nnt) {
                const uint2 b = bk[(static_cast<int64_t>(nt) * nkb + j) * 32];
                mma_16816(acc[nt], a, b.x, b.y);
                if (GATED) mma_16816(accg[nt], ag, b.x, b.y);
              }
            }
            const bool gend = GB <= 4 ? ((j + 1) % GB == 0) : (j == 3 && (c & 1));
            if (gend) {
              const int gl = (c * 4 + j) / GB, grp = g0 + gl;
              float s0, b0, s1, b1;
              sb_decode(sbu[gl * 16], A.s_dt, s0, b0);
              sb_decode(sbu[gl * 16 + 8], A.s_dt, s1, b1);
              float sg0 = 0.f, bg0 = 0.f, sg1 = 0.f, bg1 = 0.f;
              if (GATED) {
                sb_decode(sbg[gl * 16], A.s_dt, sg0, bg0);
                sb_decode(sbg[gl * 16 + 8], A.s_dt, sg1, bg1);
              }
#pragma unroll
              for (int nt = 0; nt < NTP; ++nt) {
                if (nt < nnt) {
                  const float xv = xsl[nt * 4 * ngx + grp];
                  const float r0 = fmaf(-128.f, xv, acc[nt][0] + acc[nt][1]);
                  const float r1 = fmaf(-128.f, xv, acc[nt][2] + acc[nt][3]);
                  y[nt][0] = fmaf(s0, r0, fmaf(b0, xv, y[nt][0]));
                  y[nt][1] = fmaf(s1, r1, fmaf(b1, xv, y[nt][1]));
                  if (GATED) {
                    const float q0 = fmaf(-128.f, xv, accg[nt][0] + accg[nt][1]);
                    const float q1 = fmaf(-128.f, xv, accg[nt][2] + accg[nt][3]);
                    yg[nt][0] = fmaf(sg0, q0, fmaf(bg0, xv, yg[nt][0]));
                    yg[nt][1] = fmaf(sg1, q1, fmaf(bg1, xv, yg[nt][1]));
                  }
                }
              }
            }
          }
          }
        }
      }
      __syncwarp();   // every lane has read the stage
      if (lane == 0 && ok && iss_seg < total) issue_next();
      if (++cs == NS) { cs = 0; phase ^= 1u; }
     }
     // The slot's partial sums: each warp stores its part of K; the slot's
     // first warp adds them in the fixed order ks = 0, 1, ... (double buffered
     // by tile parity, so one barrier per tile suffices).
     if (KS > 1) {
       float* rb = red + (static_cast<size_t>((ti & 1) * EM_WARPS + warp) * (4 * NTP)) * 32 + lane;
#pragma unroll
       for (int nt = 0; nt < NTP; ++nt) {
         rb[(4 * nt + 0) * 32] = y[nt][0];
         rb[(4 * nt + 1) * 32] = y[nt][1];
         rb[(4 * nt + 2) * 32] = yg[nt][0];
         rb[(4 * nt + 3) * 32] = yg[nt][1];
       }
       asm volatile("bar.sync %0, %1;" ::"r"(1 + slot), "r"(KS * 32) : "memory");
       if (ks == 0) {
         const float* r0 = red + (static_cast<size_t>((ti & 1) * EM_WARPS + slot * KS) * (4 * NTP)) * 32 + lane;
#pragma unroll
         for (int nt = 0; nt < NTP; ++nt) {
           y[nt][0] = r0[(4 * nt + 0) * 32];
           y[nt][1] = r0[(4 * nt + 1) * 32];
           yg[nt][0] = r0[(4 * nt + 2) * 32];
           yg[nt][1] = r0[(4 * nt + 3) * 32];
         }
         for (int k2 = 1; k2 < KS; ++k2) {
           const float* rk = r0 + static_cast<size_t>(k2) * (4 * NTP) * 32;
#pragma unroll
           for (int nt = 0; nt < NTP; ++nt) {
             y[nt][0] += rk[(4 * nt + 0) * 32];
             y[nt][1] += rk[(4 * nt + 1) * 32];
             yg[nt][0] += rk[(4 * nt + 2) * 32];
             yg[nt][1] += rk[(4 * nt + 3) * 32];
           }
         }
       }
     }
     if (ok && ks == 0) {
       // the tile's outputs: pair nt * 4 + t, rows 16 rt + g and + 8
#pragma unroll
       for (int nt = 0; nt < NTP; ++nt) {
         const int pl = nt * 4 + t;
         if (nt < nnt && pl < npp) {
           const int pid = s_pid[pl];
           if (pid >= 0) {
             float* o = A.out + static_cast<int64_t>(pid) * A.n_rows + rt * 16 + g;
             o[0] = (A.act >= 0) ? act_fn(A.act, yg[nt][0], y[nt][0]) : y[nt][0];
             o[8] = (A.act >= 0) ? act_fn(A.act, yg[nt][1], y[nt][1]) : y[nt][1];
           }
         }
       }
     }
    }
    // The down projection's combine, per 16-row tile: every segment's CTAs
    // count each tile they finished; the CTA that completes a tile's count
    // (nseg: one per segment) writes its combined rows for all T tokens.
    if (A.comb) {
      __threadfence();
      __syncthreads();
      for (int c0 = tb; c0 < te; c0 += EM_NT) {
        // count this segment's tiles; the ones this CTA completed go to a list,
        // and their rows x T tokens are combined by all threads in one pass
        if (threadIdx.x == 0) s_seg[0] = 0;
        __syncthreads();
        const int tt = c0 + static_cast<int>(threadIdx.x);
        if (tt < te && atomicAdd(A.ccnt + tt, 1) == nseg - 1) s_cflag[atomicAdd(&s_seg[0], 1)] = tt;
        __syncthreads();
        const int nf = s_seg[0];
        if (nf) {
          __threadfence();
          for (int i = threadIdx.x; i < nf * A.T * 16; i += EM_NT) {
            const int f = i / (A.T * 16), r = i - f * (A.T * 16);
            expert_combine_one(A, r >> 4, s_cflag[f] * 16 + (r & 15));
          }
          __syncthreads();
          if (threadIdx.x < nf) A.ccnt[s_cflag[threadIdx.x]] = 0;
        }
        __syncthreads();
      }
    }
  }
  if (!waited) griddep_wait();
  cta_stamp(A.trace, 2);
  if (!ok && lane == 0) {
    // after a wait ran out: let this warp's copies in flight land (bounded)
    // before the CTA's shared memory is released
    for (int j = gi_fail; j < issued; ++j)
      (void)eb_wait(eb_smem(bars + j % NS), static_cast<uint32_t>(j / NS) & 1u);
  }
  cta_stamp(A.trace, 3);
}

// ---------------------------------------------------------------------------
// create-time re-layouts for k_expert_mma
// ---------------------------------------------------------------------------

// Codes [E, rows, K/8] (eight 4-bit codes a word, lowest nibble first) ->
// [E, rows/16, K/64, 32 lanes, 4 words]: word j of lane (g, t) in the
// (16-row tile, 64-column chunk) holds the codes of block j (columns
// 16 j .. 16 j + 15 of the chunk) that lane needs, nibble i =
//   i = 0, 4: row g,     columns t, t + 4        i = 1, 5: row g + 8, columns t, t + 4
//   i = 2, 6: row g,     columns t + 8, t + 12   i = 3, 7: row g + 8, columns t + 8, t + 12
// (i < 4 the first column of each pair, i >= 4 the second).
static __global__ void k_tile_codes(const uint32_t* __restrict__ in, uint32_t* __restrict__ out, int E,
                                    int rows, int K) {
  const int nkc = K >> 6, words_row = K >> 3;
  const int64_t n = static_cast<int64_t>(E) * (rows >> 4) * nkc * 128;
  for (int64_t i = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x; i < n;
       i += static_cast<int64_t>(gridDim.x) * blockDim.x) {
    const int j = static_cast<int>(i & 3), lane = static_cast<int>((i >> 2) & 31);
    const int64_t r = i >> 7;   // (e, tile, kc)
    const int kc = static_cast<int>(r % nkc);
    const int64_t et = r / nkc;   // e * rows/16 + tile
    const int g = lane >> 2, t = lane & 3;
    const int64_t row0 = et * 16 + g, row1 = row0 + 8;
    const int k0 = kc * 64 + 16 * j;
    auto code = [&](int64_t row, int k) -> uint32_t {
      return (in[row * words_row + (k >> 3)] >> (4 * (k & 7))) & 0xFu;
    };
    const uint32_t w = code(row0, k0 + t) | (code(row1, k0 + t) << 4) | (code(row0, k0 + 8 + t) << 8) |
                       (code(row1, k0 + 8 + t) << 12) | (code(row0, k0 + t + 4) << 16) |
                       (code(row1, k0 + t + 4) << 20) | (code(row0, k0 + 12 + t) << 24) |
                       (code(row1, k0 + 12 + t) << 28);
    out[i] = w;
  }
}

// Scale/bias words [E, rows, K/G] -> [E, rows/16, K/G, 16]: a tile's words of
// one group are contiguous.
// MXFP4: the two E8M0 bytes of a row's 64-column chunk as one 16-bit entry,
// [E, rows, K/64] -> [E, rows/16, K/64, 16] (a tile's entries of one chunk
// contiguous, 32 bytes)
static __global__ void k_tile_sb16(const uint16_t* __restrict__ in, uint16_t* __restrict__ out, int E, int rows,
                                   int nch) {
  const int64_t n = static_cast<int64_t>(E) * rows * nch;
  for (int64_t i = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x; i < n;
       i += static_cast<int64_t>(gridDim.x) * blockDim.x) {
    const int rr = static_cast<int>(i & 15);
    const int64_t r = i >> 4;   // (e, tile, chunk)
    const int ch = static_cast<int>(r % nch);
    const int64_t et = r / nch;
    out[i] = in[(et * 16 + rr) * nch + ch];
  }
}

static __global__ void k_tile_sb(const uint32_t* __restrict__ in, uint32_t* __restrict__ out, int E, int rows,
                                 int ngr) {
  const int64_t n = static_cast<int64_t>(E) * rows * ngr;
  for (int64_t i = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x; i < n;
       i += static_cast<int64_t>(gridDim.x) * blockDim.x) {
    const int rr = static_cast<int>(i & 15);
    const int64_t r = i >> 4;   // (e, tile, grp)
    const int grp = static_cast<int>(r % ngr);
    const int64_t et = r / ngr;
    out[i] = in[(et * 16 + rr) * ngr + grp];
  }
}

}  // namespace moe
