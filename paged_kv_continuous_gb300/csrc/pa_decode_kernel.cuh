// Paged GQA decode attention (koas-w, "errors and solutions", section
// "自写 Triton Kernel", Decode_Paged_GQAAttention_Kernel: the kernel walks the
// block_table itself, keeps an online softmax and serves all query heads of
// a GQA group from one K/V read; no gather into contiguous memory) with
// flash-decoding split-K partials.
//
// Work partition.  The blocks of all sequences, in order, form one list of
// N blocks; CTA c of S takes blocks [floor(cN/S), floor((c+1)N/S)).  Every
// CTA moves the same number of bytes however skewed the lengths are, and
// consecutive sequences flow through one CTA's pipeline without draining it.
// A "piece" is the run of one sequence's blocks inside one CTA.  A piece
// that is the whole sequence writes the output rows; a cut piece writes a
// partial (o normalised over its keys, natural-log sum-exp) to the
// workspace for the merge kernel.
//
// CTA layout (288 threads).  Warp 0, lane 0 is the producer: it walks the
// CTA's block list and bulk-copies (TMA, cp.async.bulk) each physical block
// of K and V -- one contiguous [16][Hkv][128] bf16 page each -- plus the
// sequence's q row at the start of a piece, into a ring of NST stages
// guarded by full/empty mbarriers.  Warps 1..8 consume every stage; a
// half-warp unit owns one kv head g and a fixed subset of the block's 16
// tokens, lane l owns dims 8l..8l+7.  Scores are dot products in packed fp32
// (FFMA2) reduced with warp shuffles; each unit keeps a running max, sum and
// output for the G query heads of its kv head; units of the same kv head are
// merged through shared memory at the end of each piece.
#pragma once

#include "pa_common.cuh"

namespace pa {

struct DecodeParams {
  void *out;
  int out_f32;
  const uint16_t *q;        // [B][HQ][128]
  const uint16_t *k_cache;  // [num_blocks][16][HKV][128]
  const uint16_t *v_cache;
  long long num_blocks;
  const int32_t *block_tables;
  long long bt_stride;
  const int32_t *context_lens;
  int batch;
  float qk_scale_log2;  // softmax scale * log2(e): scores are kept in base 2
  int num_splits;
  float *part_o;    // [S][2][HQ][128]
  float *part_lse;  // [S][2][HQ], natural log
  int32_t *err;
};

constexpr int kDecodeConsumerWarps = 8;
constexpr int kDecodeThreads = 32 * (1 + kDecodeConsumerWarps);
constexpr int kDecodeSmemBudget = 227 * 1024;

__host__ __device__ constexpr int align_up(int x, int a) { return (x + a - 1) / a * a; }

template <int G, int HKV>
struct DecodeShape {
  static constexpr int HQ = G * HKV;
  static constexpr int KV_BYTES = kBlockSize * HKV * kHeadDim * 2;  // one page of K (or V)
  static constexpr int Q_BYTES = HQ * kHeadDim * 2;
  static constexpr int STAGE_BYTES = align_up(2 * KV_BYTES + Q_BYTES, 128);
  static constexpr int WARPS_PER_HEAD = kDecodeConsumerWarps / HKV;
  // per consumer warp: m, l and o[128] for each of its G heads
  static constexpr int RED_FLOATS_PER_HEAD = kHeadDim + 2;
  static constexpr int RED_BYTES =
      WARPS_PER_HEAD > 1 ? kDecodeConsumerWarps * G * RED_FLOATS_PER_HEAD * 4 : 0;
  static constexpr int CTL_BYTES = 256;
  static constexpr int NST_FIT = (kDecodeSmemBudget - RED_BYTES - CTL_BYTES) /
                                 (STAGE_BYTES + 16);
  static constexpr int NST = NST_FIT > 16 ? 16 : NST_FIT;
  static constexpr int SMEM = NST * STAGE_BYTES + RED_BYTES + NST * 16 + CTL_BYTES;
  static_assert(NST >= 2, "stage does not fit twice in shared memory");
  static_assert(16 % HKV == 0 && kDecodeConsumerWarps % HKV == 0, "unsupported kv heads");
};

struct DecodeCtl {
  unsigned long long total;  // N, blocks of all sequences
  long long first_prefix;    // global index of block 0 of first_b
  int first_b;               // sequence holding this CTA's first block
  int abort;                 // set by a wait that gave up
};

__device__ __forceinline__ int seq_blocks(const int32_t *ctx, int b) {
  const int n = __ldg(ctx + b);
  return n > 0 ? ceil_div_blocks(n) : 0;
}

// Online-softmax state of one half-warp unit for its G heads; lane l holds
// output dims 8l..8l+7 as four packed pairs.
template <int G>
struct UnitState {
  float2 o[G][4];
  float m[G];
  float l[G];
  __device__ __forceinline__ void reset() {
#pragma unroll
    for (int h = 0; h < G; ++h) {
      m[h] = -INFINITY;
      l[h] = 0.f;
#pragma unroll
      for (int i = 0; i < 4; ++i) o[h][i] = make_float2(0.f, 0.f);
    }
  }
};

template <int G, int HKV>
__global__ void __launch_bounds__(kDecodeThreads, 1) decode_kernel(const DecodeParams p) {
  using S = DecodeShape<G, HKV>;
  extern __shared__ __align__(128) uint8_t smem[];
  float *red = reinterpret_cast<float *>(smem + S::NST * S::STAGE_BYTES);
  uint64_t *full = reinterpret_cast<uint64_t *>(smem + S::NST * S::STAGE_BYTES + S::RED_BYTES);
  uint64_t *empty = full + S::NST;
  DecodeCtl *ctl = reinterpret_cast<DecodeCtl *>(empty + S::NST);
  volatile int *abort_flag = &ctl->abort;

  const int tid = threadIdx.x;
  const int warp = tid >> 5;
  const int lane = tid & 31;
  const long long nsplit = p.num_splits;
  const long long c = blockIdx.x;

  // ---- 1. total block count N and this CTA's block range --------------------
  if (tid == 0) {
    ctl->total = 0;
    ctl->first_b = -1;
    ctl->first_prefix = 0;
    ctl->abort = 0;
  }
  __syncthreads();
  {
    unsigned long long local = 0;
    for (int b = tid; b < p.batch; b += blockDim.x) local += seq_blocks(p.context_lens, b);
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) local += __shfl_xor_sync(0xffffffffu, local, off);
    if (lane == 0 && local) atomicAdd(&ctl->total, local);
  }
  __syncthreads();
  const long long N = (long long)ctl->total;
  const long long lo = N ? split_begin(c, nsplit, N) : 0;
  const long long hi = N ? split_begin(c + 1, nsplit, N) : 0;

  // ---- 2. block-wide scan of sequence block counts: find the sequence that
  //         holds block `lo`; zero the rows of empty sequences this CTA owns.
  {
    __shared__ long long warp_tot[kDecodeThreads / 32];
    long long running = 0;
    for (int base = 0; base < p.batch; base += blockDim.x) {
      const int b = base + tid;
      const int n = b < p.batch ? seq_blocks(p.context_lens, b) : 0;
      long long incl = n;
#pragma unroll
      for (int off = 1; off < 32; off <<= 1) {
        const long long y = __shfl_up_sync(0xffffffffu, incl, off);
        if (lane >= off) incl += y;
      }
      if (lane == 31) warp_tot[warp] = incl;
      __syncthreads();
      long long before = running;
      for (int w = 0; w < warp; ++w) before += warp_tot[w];
      long long chunk_total = 0;
      for (int w = 0; w < (int)(blockDim.x >> 5); ++w) chunk_total += warp_tot[w];
      const long long prefix = before + incl - n;  // global index of block 0 of b
      if (b < p.batch) {
        if (n > 0 && prefix <= lo && lo < prefix + n && lo < hi) {
          ctl->first_b = b;
          ctl->first_prefix = prefix;
        }
        const bool owns_empty =
            n == 0 && ((lo <= prefix && prefix < hi) || (prefix >= N && c == nsplit - 1));
        if (owns_empty) {
          const long long row0 = (long long)b * S::HQ * kHeadDim;
          if (p.out_f32) {
            float *o = static_cast<float *>(p.out) + row0;
            for (int i = 0; i < S::HQ * kHeadDim; ++i) o[i] = 0.f;
          } else {
            uint16_t *o = static_cast<uint16_t *>(p.out) + row0;
            for (int i = 0; i < S::HQ * kHeadDim; ++i) o[i] = 0;
          }
        }
      }
      running += chunk_total;
      __syncthreads();
    }
  }
  if (lo >= hi) return;  // no block for this CTA (N < S)
  if (ctl->first_b < 0) {  // cannot happen for consistent inputs; never walk from b = -1
    if (tid == 0) report(p.err, PA_DEVERR_SHAPE);
    return;
  }

  // ---- 3. pipeline barriers -------------------------------------------------
  const uint32_t stage0 = smem_addr(smem);
  const uint32_t full0 = smem_addr(full);
  const uint32_t empty0 = smem_addr(empty);
  if (tid == 0) {
    for (int i = 0; i < S::NST; ++i) {
      mbar_init(full0 + 8 * i, 1);
      mbar_init(empty0 + 8 * i, kDecodeConsumerWarps);
    }
    fence_barrier_init();
  }
  __syncthreads();
  const int first_b = ctl->first_b;
  const long long first_prefix = ctl->first_prefix;

  if (warp == 0) {
    // ---- 4. producer ---------------------------------------------------------
    if (lane != 0) return;
    const uint64_t pol_kv = l2_policy_evict_first();
    const uint64_t pol_q = l2_policy_evict_last();
    int b = first_b;
    int n = seq_blocks(p.context_lens, b);
    int j = (int)(lo - first_prefix);
    long long issued = 0;
    for (long long gb = lo; gb < hi; ++gb, ++issued, ++j) {
      if (j == n) {
        do {
          ++b;
          n = seq_blocks(p.context_lens, b);
        } while (n == 0);
        j = 0;
      }
      const int st = (int)(issued % S::NST);
      const int round = (int)(issued / S::NST);
      if (round > 0 && !mbar_wait(empty0 + 8 * st, (round - 1) & 1, abort_flag, p.err)) break;
      const bool piece_first = (gb == lo) || (j == 0);
      // a row holds bt_stride entries: a context longer than the row is a
      // caller error, reported and not read
      const bool in_row = j < p.bt_stride;
      const long long phys = in_row ? __ldg(p.block_tables + (long long)b * p.bt_stride + j) : -1;
      const bool ok = phys >= 0 && phys < p.num_blocks;
      const uint32_t bytes = (ok ? 2u * S::KV_BYTES : 0u) + (piece_first ? S::Q_BYTES : 0u);
      const uint32_t dst = stage0 + st * S::STAGE_BYTES;
      const uint32_t bar = full0 + 8 * st;
      mbar_arrive_expect_tx(bar, bytes);
      if (ok) {
        const long long off = phys * (long long)(kBlockSize * HKV * kHeadDim);
        bulk_load(dst, p.k_cache + off, S::KV_BYTES, bar, pol_kv);
        bulk_load(dst + S::KV_BYTES, p.v_cache + off, S::KV_BYTES, bar, pol_kv);
      } else {
        report(p.err, in_row ? PA_DEVERR_BLOCK_INDEX : PA_DEVERR_SHAPE);
      }
      if (piece_first)
        bulk_load(dst + 2 * S::KV_BYTES, p.q + (long long)b * S::HQ * kHeadDim, S::Q_BYTES, bar,
                  pol_q);
    }
    if (*abort_flag) {
      // Drain: copies still in flight must land before the CTA's shared
      // memory is released.  Bounded, independent of the abort flag.
      volatile int never = 0;
      const long long from = issued > S::NST ? issued - S::NST : 0;
      for (long long i = from; i < issued; ++i)
        mbar_wait(full0 + 8 * (int)(i % S::NST), (int)((i / S::NST) & 1), &never, nullptr);
    }
    return;
  }

  // ---- 5. consumers -----------------------------------------------------------
  const int cw = warp - 1;                   // consumer warp 0..7
  const int hw = lane >> 4;                  // half-warp
  const int l = lane & 15;                   // dims 8l..8l+7
  const int g = cw % HKV;                    // kv head of this warp
  constexpr int SUBS = kBlockSize / HKV;     // units per kv head = token stride
  const int sub = (cw / HKV) * 2 + hw;       // tokens sub, sub + SUBS, ...
  const int row_off = g * kHeadDim * 2 + l * 16;  // byte offset of (g, 8l) in a token row

  UnitState<G> st;
  st.reset();
  float2 qf[G][4];

  int b = first_b;
  int n = seq_blocks(p.context_lens, b);
  int ctx = __ldg(p.context_lens + b);
  int j = (int)(lo - first_prefix);
  int piece_j0 = j;
  long long it = 0;
  for (long long gb = lo; gb < hi; ++gb, ++it, ++j) {
    if (j == n) {
      do {
        ++b;
        ctx = __ldg(p.context_lens + b);
        n = ctx > 0 ? ceil_div_blocks(ctx) : 0;
      } while (n == 0);
      j = 0;
    }
    const bool piece_first = (gb == lo) || (j == 0);
    const bool piece_last = (gb == hi - 1) || (j == n - 1);
    const int sidx = (int)(it % S::NST);
    const uint32_t sbase = stage0 + sidx * S::STAGE_BYTES;
    // warp-uniform: the shuffles below need every lane of the warp
    const bool have = __all_sync(
        0xffffffffu, mbar_wait(full0 + 8 * sidx, (int)((it / S::NST) & 1), abort_flag, p.err));
    if (piece_first) {
      piece_j0 = j;
      st.reset();
      if (have) {
#pragma unroll
        for (int h = 0; h < G; ++h) {
          const uint4 w = lds128(sbase + 2 * S::KV_BYTES + (g * G + h) * kHeadDim * 2 + l * 16);
          const uint32_t ws[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
          for (int i = 0; i < 4; ++i) {
            const float2 f = bf16x2_to_float2(ws[i]);
            qf[h][i] = make_float2(f.x * p.qk_scale_log2, f.y * p.qk_scale_log2);
          }
        }
      }
    }
    const int valid = min(kBlockSize, ctx - j * kBlockSize);  // keys of this block
    // Both half-warps enter together whenever the warp's first token is a key
    // (the shuffles need all 32 lanes); tokens past `valid` are masked.
    if (have && (cw / HKV) * 2 < valid) {
      // scores of this unit's tokens, all G heads, partial over 8 dims
      float s[HKV][G];
#pragma unroll
      for (int t = 0; t < HKV; ++t) {
        const int tok = sub + t * SUBS;
        const uint4 w = lds128(sbase + tok * HKV * kHeadDim * 2 + row_off);
        const float2 k0 = bf16x2_to_float2(w.x), k1 = bf16x2_to_float2(w.y);
        const float2 k2 = bf16x2_to_float2(w.z), k3 = bf16x2_to_float2(w.w);
#pragma unroll
        for (int h = 0; h < G; ++h) {
          float2 a = __fmul2_rn(qf[h][0], k0);
          a = __ffma2_rn(qf[h][1], k1, a);
          a = __ffma2_rn(qf[h][2], k2, a);
          a = __ffma2_rn(qf[h][3], k3, a);
          s[t][h] = a.x + a.y;
        }
      }
#pragma unroll
      for (int t = 0; t < HKV; ++t)
#pragma unroll
        for (int h = 0; h < G; ++h)
#pragma unroll
          for (int off = 8; off > 0; off >>= 1)
            s[t][h] += __shfl_xor_sync(0xffffffffu, s[t][h], off);
      // online softmax update (base 2; q was pre-scaled by scale*log2 e)
#pragma unroll
      for (int h = 0; h < G; ++h) {
        float mx = -INFINITY;
#pragma unroll
        for (int t = 0; t < HKV; ++t)
          if (sub + t * SUBS < valid) mx = fmaxf(mx, s[t][h]);
        const float m_new = fmaxf(st.m[h], mx);
        // no key seen yet by this unit (all masked so far): state stays empty
        const float alpha = m_new == -INFINITY ? 1.f : exp2f(st.m[h] - m_new);
        st.m[h] = m_new;
        float lsum = st.l[h] * alpha;
#pragma unroll
        for (int t = 0; t < HKV; ++t) {
          const float pt = (sub + t * SUBS < valid) ? exp2f(s[t][h] - m_new) : 0.f;
          s[t][h] = pt;
          lsum += pt;
        }
        st.l[h] = lsum;
        const float2 a2 = make_float2(alpha, alpha);
#pragma unroll
        for (int i = 0; i < 4; ++i) st.o[h][i] = __fmul2_rn(st.o[h][i], a2);
      }
      // o += p v
#pragma unroll
      for (int t = 0; t < HKV; ++t) {
        const int tok = sub + t * SUBS;
        if (tok < valid) {
          const uint4 w = lds128(sbase + S::KV_BYTES + tok * HKV * kHeadDim * 2 + row_off);
          const float2 v0 = bf16x2_to_float2(w.x), v1 = bf16x2_to_float2(w.y);
          const float2 v2 = bf16x2_to_float2(w.z), v3 = bf16x2_to_float2(w.w);
#pragma unroll
          for (int h = 0; h < G; ++h) {
            const float2 pp = make_float2(s[t][h], s[t][h]);
            st.o[h][0] = __ffma2_rn(pp, v0, st.o[h][0]);
            st.o[h][1] = __ffma2_rn(pp, v1, st.o[h][1]);
            st.o[h][2] = __ffma2_rn(pp, v2, st.o[h][2]);
            st.o[h][3] = __ffma2_rn(pp, v3, st.o[h][3]);
          }
        }
      }
    }
    __syncwarp();
    if (lane == 0) mbar_arrive(empty0 + 8 * sidx);

    if (!piece_last) continue;
    // ---- end of a piece: merge units, write output row or partial ----------
    const bool head_cut = piece_j0 > 0;
    const bool tail_cut = j < n - 1;
    const bool whole = !head_cut && !tail_cut;
    // merge the two half-warps (same kv head, disjoint tokens)
#pragma unroll
    for (int h = 0; h < G; ++h) {
      const float mo = __shfl_xor_sync(0xffffffffu, st.m[h], 16);
      const float lo_ = __shfl_xor_sync(0xffffffffu, st.l[h], 16);
      const float M = fmaxf(st.m[h], mo);
      const float wa = st.m[h] == -INFINITY ? 0.f : exp2f(st.m[h] - M);
      const float wb = mo == -INFINITY ? 0.f : exp2f(mo - M);
      st.l[h] = st.l[h] * wa + lo_ * wb;
      st.m[h] = M;
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        float2 x = st.o[h][i];
        float2 y;
        y.x = __shfl_xor_sync(0xffffffffu, x.x, 16);
        y.y = __shfl_xor_sync(0xffffffffu, x.y, 16);
        st.o[h][i] = make_float2(x.x * wa + y.x * wb, x.y * wa + y.y * wb);
      }
    }
    const long long slot_row = (c * 2 + (head_cut ? 0 : 1)) * S::HQ;
    if constexpr (S::WARPS_PER_HEAD == 1) {
      if (hw == 0) {
#pragma unroll
        for (int h = 0; h < G; ++h) {
          const int qh = g * G + h;
          const float L = st.l[h];
          const float inv = L > 0.f ? 1.f / L : 0.f;
          float r[8];
#pragma unroll
          for (int i = 0; i < 4; ++i) {
            r[2 * i] = st.o[h][i].x * inv;
            r[2 * i + 1] = st.o[h][i].y * inv;
          }
          if (whole) {
            const long long base = ((long long)b * S::HQ + qh) * kHeadDim + l * 8;
            if (p.out_f32) {
              float4 *o4 = reinterpret_cast<float4 *>(static_cast<float *>(p.out) + base);
              o4[0] = make_float4(r[0], r[1], r[2], r[3]);
              o4[1] = make_float4(r[4], r[5], r[6], r[7]);
            } else {
              uint4 w;
              w.x = float2_to_bf16x2(r[0], r[1]);
              w.y = float2_to_bf16x2(r[2], r[3]);
              w.z = float2_to_bf16x2(r[4], r[5]);
              w.w = float2_to_bf16x2(r[6], r[7]);
              *reinterpret_cast<uint4 *>(static_cast<uint16_t *>(p.out) + base) = w;
            }
          } else {
            float4 *o4 = reinterpret_cast<float4 *>(p.part_o + (slot_row + qh) * kHeadDim + l * 8);
            o4[0] = make_float4(r[0], r[1], r[2], r[3]);
            o4[1] = make_float4(r[4], r[5], r[6], r[7]);
            if (l == 0)
              p.part_lse[slot_row + qh] =
                  L > 0.f ? (st.m[h] + __log2f(L)) * 0.69314718055994531f : -INFINITY;
          }
        }
      }
    } else {
      // several warps hold the same kv head: combine through shared memory
      if (hw == 0) {
#pragma unroll
        for (int h = 0; h < G; ++h) {
          float *r = red + (cw * G + h) * S::RED_FLOATS_PER_HEAD;
          if (l == 0) {
            r[0] = st.m[h];
            r[1] = st.l[h];
          }
          // r + 2 is 8-byte aligned (130 floats per head record): float2 stores
          float2 *o2 = reinterpret_cast<float2 *>(r + 2 + l * 8);
#pragma unroll
          for (int i = 0; i < 4; ++i) o2[i] = st.o[h][i];
        }
      }
      named_barrier(1, kDecodeConsumerWarps * 32);
      const int ct = tid - 32;
      for (int e = ct * 2; e < S::HQ * kHeadDim; e += kDecodeConsumerWarps * 32 * 2) {
        const int qh = e / kHeadDim;
        const int d = e % kHeadDim;
        const int gh = qh / G;
        const int h = qh % G;
        float M = -INFINITY;
#pragma unroll
        for (int k = 0; k < S::WARPS_PER_HEAD; ++k)
          M = fmaxf(M, red[((gh + k * HKV) * G + h) * S::RED_FLOATS_PER_HEAD]);
        float L = 0.f, o0 = 0.f, o1 = 0.f;
#pragma unroll
        for (int k = 0; k < S::WARPS_PER_HEAD; ++k) {
          const float *r = red + ((gh + k * HKV) * G + h) * S::RED_FLOATS_PER_HEAD;
          const float w = r[0] == -INFINITY ? 0.f : exp2f(r[0] - M);
          L += r[1] * w;
          o0 += r[2 + d] * w;
          o1 += r[3 + d] * w;
        }
        const float inv = L > 0.f ? 1.f / L : 0.f;
        o0 *= inv;
        o1 *= inv;
        if (whole) {
          const long long base = ((long long)b * S::HQ + qh) * kHeadDim + d;
          if (p.out_f32)
            *reinterpret_cast<float2 *>(static_cast<float *>(p.out) + base) = make_float2(o0, o1);
          else
            *reinterpret_cast<uint32_t *>(static_cast<uint16_t *>(p.out) + base) =
                float2_to_bf16x2(o0, o1);
        } else {
          *reinterpret_cast<float2 *>(p.part_o + (slot_row + qh) * kHeadDim + d) =
              make_float2(o0, o1);
          if (d == 0)
            p.part_lse[slot_row + qh] =
                L > 0.f ? (M + __log2f(L)) * 0.69314718055994531f : -INFINITY;
        }
      }
      named_barrier(1, kDecodeConsumerWarps * 32);
    }
  }
}

// Launches decode_kernel<G, HKV> for one G (defined per HKV in pa_decode_h*.cu).
template <int HKV>
cudaError_t launch_decode(int G, const DecodeParams &p, cudaStream_t s, int device);
template <int HKV>
int decode_smem_bytes(int G);

}  // namespace pa
