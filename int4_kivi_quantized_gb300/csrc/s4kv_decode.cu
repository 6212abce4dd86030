// Read side of the cache: paged decode attention over the int4 history plus
// the full-precision residual ("4.4 KV Cache 量化", section 2: P = softmax(QK^T
// / sqrt d), output PV; section 3.2: residual and history both take part).
//
// One kernel per call, every warp an independent worker. The (sequence, kv head)
// segments are laid end to end on a cost line (one unit per 32-token key group,
// more per tail chunk) that is cut into one contiguous slice per warp. A warp
// streams its key groups through a two-stage ring in shared memory: both page
// records of a group (3 KiB each: codes and fp32 metadata of one kv head)
// arrive by 1-D bulk TMA, guarded by an mbarrier with a bounded wait. Nothing
// restored goes back to HBM ("给 KV cache 减肥", section 3.1: restore when the
// query reads):
//  * tensor-core path: the per-channel key scale is folded into the query
//    (q'_c = q_c s_c, one f16x2 operand per 16-channel slice) and the key min
//    into a per-head bias; nibbles are unpacked to f16 with the magic-number
//    method (integer OR into the mantissa of 1024.0, then subtract) and fed to
//    mma.sync m16n8k16 with tokens as rows and GQA heads as columns. The value
//    side folds the per-token scale into the probabilities (p'_t = p_t s_tk) and
//    the value min into a per-head, per-group bias, with channels as rows.
//  * FFMA path: the same staging with CUDA-core arithmetic, for comparison.
// Tokens past the last group quantized for both keys and values (at most
// R + 31) go through a per-token path that reads the rings. A segment inside
// one warp's slice is written directly; a segment split between warps leaves
// one (m, l, o) partial per warp, and merge_kernel, launched right behind as a
// programmatic dependent, combines them with the log-sum-exp rule. FP8 pages
// take their own main loop (single-page stages, no rings).

#include "s4kv_kernels.cuh"
#include "s4kv_quant.cuh"

namespace s4kv {
namespace {

// ---- decode step: the append of one token per sequence, inside the launch ----
// Every warp of the grid takes (sequence, kv head) items: it checks the stored
// length, quantizes the value token that leaves the window into its page (from
// the ring row it is about to overwrite), writes the new rows into the rings,
// and quantizes the key group the new token completes (from the ring rows and
// the new row). The same quantizer as the append kernels, so the pages and
// rings are those a separate append would leave. FP8 pages take the token
// straight into its page.
template <int BITS>
__device__ __forceinline__ void step_append(const DecodeArgs& a, int gw, int nwarps) {
  const int lane = threadIdx.x & 31;
  for (int it = gw; it < a.B * a.H; it += nwarps) {
    const int b = it / a.H, h = it - (it / a.H) * a.H;
    const int T1 = a.seq_lens[b], T0 = T1 - 1;
    const int slot = a.slot_ids ? a.slot_ids[b] : b;
    if (T1 <= 0 || T1 > a.max_seq_len) {
      if (lane == 0) report(a.status, S4KV_ERR_DEVICE, S4KV_DEV_BAD_LENGTH, b);
      continue;
    }
    if (slot < 0 || slot >= a.max_slots) {
      if (lane == 0) report(a.status, S4KV_ERR_DEVICE, S4KV_DEV_BAD_SLOT, slot);
      continue;
    }
    if (static_cast<long long>(a.bt_stride) * kP < T1) {
      if (lane == 0) report(a.status, S4KV_ERR_DEVICE, S4KV_DEV_BAD_TABLE, b);
      continue;
    }
    int* lw = a.lens_w + slot * a.H + h;
    const int stored = __ldcg(lw);
    if (T0 != 0 && stored != T0) {
      if (lane == 0) report(a.status, S4KV_ERR_DEVICE, S4KV_DEV_BAD_LENGTH, b);
      continue;
    }
    const int* bt_row = a.block_table + static_cast<long long>(b) * a.bt_stride;
    const long long row = (static_cast<long long>(b) * a.H + h) * kD;
    const uint2 kr = reinterpret_cast<const uint2*>(a.knew + row)[lane];
    const uint2 vr = reinterpret_cast<const uint2*>(a.vnew + row)[lane];
    auto record = [&](int logical_page) -> char* {
      const int pp = bt_row[logical_page];
      if (pp < 0 || pp >= a.num_pages) {
        if (lane == 0) report(a.status, S4KV_ERR_DEVICE, S4KV_DEV_BAD_PAGE, pp);
        return nullptr;
      }
      return const_cast<char*>(a.pages) + (static_cast<long long>(pp) * a.H + h) * Rec<BITS>::kBytes;
    };
    if constexpr (BITS == 8) {
      char* rec = record(T0 / kP);
      if (rec) quant::fp8_token(rec, T0, kr, vr, a.fp8_scale[h], a.fp8_scale[a.H + h], a.dtype);
    } else {
      uint16_t* kring = reinterpret_cast<uint16_t*>(const_cast<char*>(a.kring)) + slot * a.kring_slot + h * a.kring_head;
      uint16_t* vring = reinterpret_cast<uint16_t*>(const_cast<char*>(a.vring)) + slot * a.vring_slot + h * a.vring_head;
      if (T1 > a.R) {   // token T0 - R leaves the value window (the new token itself when R = 0)
        const int tv = T0 - a.R;
        const uint2 old = a.R > 0 ? reinterpret_cast<const uint2*>(vring + static_cast<long long>(tv % a.R) * kD)[lane] : vr;
        quant::value_token<BITS>(record(tv / kP), tv, old, a.dtype);
      }
      __syncwarp();
      if (a.R > 0) reinterpret_cast<uint2*>(vring + static_cast<long long>(T0 % a.R) * kD)[lane] = vr;
      if (T1 % kG != 0) {
        reinterpret_cast<uint2*>(kring + static_cast<long long>(T0 % kG) * kD)[lane] = kr;
      } else {   // the new token completes key group T1 / G - 1: rows T1 - G .. T1 - 1 sit in ring rows 0 .. G - 1
        uint2 rows[kG];
#pragma unroll
        for (int t = 0; t < kG - 1; ++t) rows[t] = reinterpret_cast<const uint2*>(kring + static_cast<long long>(t) * kD)[lane];
        rows[kG - 1] = kr;
        const int grp = T1 / kG - 1;
        quant::key_group<BITS>(record(2 * grp), record(2 * grp + 1), rows, a.dtype);
      }
    }
    __syncwarp();
    if (lane == 0) *lw = T1;
  }
}

// Barrier of the whole grid of a cooperative launch (every CTA is resident):
// an arrival count and a generation word in the pool's status area. The last
// CTA to arrive resets the count and advances the generation; the others wait
// for the generation to move, for at most wait_ns (then the status reads
// TIMEOUT and the kernel goes on: every address it uses is still checked).
// Writes before the barrier are visible after it to ordinary loads and, by the
// proxy fences, to bulk copies.
__device__ bool grid_sync(const DecodeArgs& a) {
  __shared__ int ok;
  asm volatile("fence.proxy.async.global;" ::: "memory");
  __syncthreads();
  if (threadIdx.x == 0) {
    unsigned* cnt = a.gbar;
    volatile unsigned* gen = a.gbar + 1;
    const unsigned g0 = *gen;
    __threadfence();
    bool done = true;
    if (atomicAdd(cnt, 1u) + 1u == gridDim.x) {
      atomicExch(cnt, 0u);
      __threadfence();
      atomicAdd(a.gbar + 1, 1u);
    } else {
      const unsigned long long t0 = global_ns();
      while (*gen == g0) {
        if (global_ns() - t0 > static_cast<unsigned long long>(a.wait_ns)) {
          done = false;
          break;
        }
        __nanosleep(64);
      }
    }
    __threadfence();
    if (!done) report(a.status, S4KV_ERR_DEVICE_TIMEOUT, S4KV_DEV_TIMEOUT, -2);
    ok = done ? 1 : 0;
  }
  __syncthreads();
  asm volatile("fence.proxy.async.global;" ::: "memory");
  return ok != 0;
}

// The merge items it0, it0 + stride, ...: one warp per (segment, query head).
// It reads the segment's merge descriptor and skips segments written directly
// (inside one warp's slice, or an invalid slot); otherwise it combines the
// partials of the segment's contributors by the log-sum-exp rule, kMC
// contributors at a time: their (m, l) pairs (lane = contributor) and rows are
// loaded together, then weighed and summed.
__device__ __forceinline__ void merge_items(const DecodeArgs& a, long long it0, long long stride,
                                       unsigned long long& tm_seg, unsigned long long& tm_ld) {
  const int lane = threadIdx.x & 31;
  const long long* desc = meta_of(a);
  const long long items = static_cast<long long>(a.B) * a.H * a.g;
  const long long pf = partial_floats(a.pcols);
  for (long long it = it0; it < items; it += stride) {
    const int j = static_cast<int>(it % a.g);
    const long long bh = it / a.g;
    const long long d = __ldcg(desc + bh);
    const int nc = static_cast<int>(d >> 32);
    if (nc <= 0) continue;   // inside one slice, or an invalid slot: written by decode_kernel
    S4KV_TRACE(tm_seg = global_ns();)
    // contributor 0 is the descriptor's slot; contributor i >= 1 is the warp i
    // places on, slot 0 (the segment is the first piece of its slice)
    const long long first = static_cast<long long>(static_cast<unsigned>(d & 0xffffffffLL));
    auto part = [&](int i) -> const float* {
      return a.ws + (i == 0 ? first : (first & ~1LL) + 2LL * i) * pf;
    };
    float M = -INFINITY, L = 0.0f;
    float4 O = make_float4(0.0f, 0.0f, 0.0f, 0.0f);
    for (int i0 = 0; i0 < nc; i0 += kMC) {
      const int nch = min(kMC, nc - i0);
      const float* W = part(i0 + (lane < nch ? lane : 0)) + a.pcols * kD + 2 * j;
      const float mi = lane < nch ? __ldcg(W) : -INFINITY;
      const float li = lane < nch ? __ldcg(W + 1) : 0.0f;
      float4 r[kMC];
#pragma unroll
      for (int u = 0; u < kMC; ++u)
        r[u] = u < nch ? __ldcg(reinterpret_cast<const float4*>(part(i0 + u) + j * kD + 4 * lane))
                       : make_float4(0.0f, 0.0f, 0.0f, 0.0f);
      S4KV_TRACE(if (!tm_ld) tm_ld = global_ns() + static_cast<unsigned long long>(r[kMC - 1].x == 12345.0f);)
      const float mn = fmaxf(M, warp_max(mi));
      const bool live = mn != -INFINITY;   // all partials empty so far: nothing to weigh
      const float ao = live ? ex2(M - mn) : 1.0f;
      const float wi = live ? ex2(mi - mn) : 0.0f;
      L = fmaf(L, ao, warp_sum(wi * li));
      O = make_float4(O.x * ao, O.y * ao, O.z * ao, O.w * ao);
#pragma unroll
      for (int u = 0; u < kMC; ++u) {
        const float w = __shfl_sync(0xffffffffu, wi, u);   // 0 for absent contributors
        O = make_float4(fmaf(w, r[u].x, O.x), fmaf(w, r[u].y, O.y), fmaf(w, r[u].z, O.z), fmaf(w, r[u].w, O.w));
      }
      M = mn;
    }
    const float inv = L > 0.0f ? 1.0f / L : 0.0f;
    store_out(a, static_cast<long long>(bh / a.H) * a.Hq + (bh % a.H) * a.g + j, lane,
              make_float4(O.x * inv, O.y * inv, O.z * inv, O.w * inv));
  }
  (void)tm_seg;
  (void)tm_ld;
}

#ifndef S4KV_STEP_MERGE
#define S4KV_STEP_MERGE 0
#endif
// The decode step merges split segments in its own launch (after a second grid
// barrier) when 1, or leaves them to merge_kernel launched behind it when 0.
constexpr bool kStepMerge = S4KV_STEP_MERGE != 0;

// STEP: the decode step's kernel (the appends, a grid barrier, the attention, a
// second grid barrier and the merge, in one cooperative launch); otherwise the
// attention alone, with merge_kernel launched behind it.
template <int IMPL, int BITS, bool STEP = false>
__global__ void __launch_bounds__(32 * warps_of<IMPL>(), IMPL != 1 ? S4KV_DECODE_MIN_CTAS : 1)
    decode_kernel(DecodeArgs a) {
  static_assert(BITS == 4 || IMPL != 1, "the FFMA path reads 4-bit records");
  // decode step: the appends of this call, then a grid barrier (first, so that
  // nothing of the attention is live across them)
  if constexpr (STEP) {
    constexpr int kW = warps_of<IMPL>();
    step_append<BITS>(a, static_cast<int>(blockIdx.x) * kW + static_cast<int>(threadIdx.x >> 5),
                      static_cast<int>(gridDim.x) * kW);
    grid_sync(a);
  }
  using F = Rec<BITS>;
  constexpr int RS = kRecStrideB<BITS>;
  constexpr int kWarps = warps_of<IMPL>();
  constexpr int kThreads = 32 * kWarps;
  using SmemT = Smem<kWarps>;
  extern __shared__ __align__(128) uint8_t smem_raw[];
  SmemT& sm = *reinterpret_cast<SmemT*>(smem_raw);
  long long* pre = reinterpret_cast<long long*>(smem_raw + prefix_offset<IMPL>());   // [B + 1]
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  uint8_t* st0 = sm.region[warp];
  uint8_t* st1 = sm.region[warp] + kStageBytesB<BITS>;
  uint64_t* bar = sm.bar[warp];
  float* ptile = sm.ptile[warp];
  float* q_s = reinterpret_cast<float*>(smem_raw + sizeof(SmemT)) + warp * 2 * kNH * kD;   // FFMA path
  float* qp = q_s + kNH * kD;   // FFMA path only

  constexpr int kNS = BITS == 8 ? kFp8Stages : kStages;   // stages of the main loop
  if (lane == 0) {
    for (int i = 0; i < kNS; ++i) mbar_init(&bar[i], 1);
  }
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  __shared__ __align__(16) uint4 zero16;   // ldmatrix source of absent value-ring rows
  if (tid == 0) zero16 = make_uint4(0u, 0u, 0u, 0u);
  const uint32_t zero_s = smem_u32(&zero16);
  // cost prefix over sequences: sequence b owns H segments of seg_cost(T_b)
  {
    long long carry = 0;
    __shared__ long long wt[kWarps];
    for (int base = 0; base < a.B; base += kThreads) {
      const int b = base + tid;
      const long long cnt = b < a.B ? a.H * seg_cost<BITS>(a.seq_lens[b], a.R, a.tail_cost).cost : 0;
      long long x = cnt;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const long long y = __shfl_up_sync(0xffffffffu, x, o);
        if (lane >= o) x += y;
      }
      if (lane == 31) wt[warp] = x;
      __syncthreads();
      long long before = carry, total = 0;
      for (int q = 0; q < kWarps; ++q) {
        if (q < warp) before += wt[q];
        total += wt[q];
      }
      if (b < a.B) pre[b] = before + x - cnt;
      __syncthreads();
      carry += total;
    }
    if (tid == 0) pre[a.B] = carry;
    __syncthreads();
  }
  const long long C = pre[a.B];
  int n_act = static_cast<int>(gridDim.x) * kWarps;
  if (a.max_warps > 0 && a.max_warps < n_act) n_act = a.max_warps;
  {
    // at least kMinUnits of work per warp: fewer partials on small problems
    const long long cap = (C + kMinUnits - 1) / kMinUnits;
    if (cap < n_act) n_act = static_cast<int>(cap);
  }
  // merge_kernel may be scheduled now; it waits for this grid to complete
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  const int gw = blockIdx.x * kWarps + warp;
  if (gw < n_act) {
    const long long r0 = gw * C / n_act, r1 = (gw + 1) * C / n_act;
    // trace words: 0 start, 1 end, 2..5 phase times (prologue, main, tail, finalize), 6 segments,
    // 7 main groups, 8..10 tail parts (scores, softmax, PV), 11 tail groups, 12 main-loop waits,
    // 13 tail waits, 14 partial stores; 15..21 unused
    S4KV_TRACE(unsigned long long tr[kTraceWords] = {};
               tr[0] = global_ns();
               int wslot = 12;
               unsigned long long tmark = tr[0];
               auto tlap = [&](int slot) { const unsigned long long t = global_ns(); tr[slot] += t - tmark; tmark = t; };)

    uint32_t phase = 0, pend = 0;   // per-stage wait parity and copies in flight (bit per stage)
    const uint64_t once = policy_evict_first();
    bool aborted = false;
    auto issue = [&](int s, int lp0, int np, const Seg& sg) {
      fence_proxy_async();   // earlier generic accesses of the buffer come first
      __syncwarp();
      if (lane == 0) {
        uint8_t* dst = s ? st1 : st0;
        mbar_expect_tx(&bar[s], np * kRec);
        for (int i = 0; i < np; ++i) bulk_load_hint(dst + i * kRecStride, rec_of(sg, lp0 + i), kRec, &bar[s], once);
      }
      pend |= 1u << s;
    };
    // both records of one key group, pool pages p0 and p1, into stage s
    auto issue_pp = [&](int s, int p0, int p1, const Seg& sg) {
      fence_proxy_async();
      __syncwarp();
      if (lane == 0) {
        uint8_t* dst = s ? st1 : st0;
        mbar_expect_tx(&bar[s], 2 * F::kBytes);
        bulk_load_hint(dst, rec_at<BITS>(sg, p0), F::kBytes, &bar[s], once);
        bulk_load_hint(dst + RS, rec_at<BITS>(sg, p1), F::kBytes, &bar[s], once);
      }
      pend |= 1u << s;
    };
    auto wait = [&](int s) -> bool {
      S4KV_TRACE(const unsigned long long tw = global_ns();)
      const bool got = mbar_wait(&bar[s], (phase >> s) & 1u, aborted ? 0 : a.wait_ns);
      S4KV_TRACE(tr[wslot] += global_ns() - tw;)
      if (!got) return false;
      phase ^= 1u << s;
      pend &= ~(1u << s);
      return true;
    };
    auto fail = [&](long long where) {   // bounded wait ran out: drain, then go on without compute
      if (lane == 0) report(a.status, S4KV_ERR_DEVICE_TIMEOUT, S4KV_DEV_TIMEOUT, static_cast<int>(where));
      aborted = true;
      for (int s = 0; s < kNS; ++s) {
        if ((pend >> s) & 1u) {
          mbar_wait(&bar[s], (phase >> s) & 1u, kDrainNs);
          phase ^= 1u << s;
          pend &= ~(1u << s);
        }
      }
    };

    // first segment touching this slice
    int b;
    {
      int lo = 0, hi = a.B - 1;
      while (lo < hi) {
        const int mid = (lo + hi + 1) >> 1;
        if (pre[mid] <= r0) lo = mid; else hi = mid - 1;
      }
      b = lo;
    }
    SegCost sc = seg_cost<BITS>(a.seq_lens[b], a.R, a.tail_cost);
    int h = static_cast<int>((r0 - pre[b]) / sc.cost);
    long long seg_start = pre[b] + h * sc.cost;

    while (seg_start < r1) {
      S4KV_TRACE(tr[6] += 1;)
      const long long seg_end = seg_start + sc.cost;
      const int T = max(a.seq_lens[b], 0);
      const long long lo = max(r0, seg_start) - seg_start, hi = min(r1, seg_end) - seg_start;
      const bool own = lo == 0 && hi == sc.cost;
      // main groups and tail chunks whose cost position starts inside [lo, hi)
      const int nm = sc.main_groups;
      const int u0 = static_cast<int>(lo < nm ? lo : nm), u1 = static_cast<int>(hi < nm ? hi : nm);
      int c0 = 0, c1 = 0;
      if (sc.tail_chunks > 0 && hi > nm) {
        c0 = static_cast<int>(lo > nm ? (lo - nm + a.tail_cost - 1) / a.tail_cost : 0);
        const long long cc = (hi - nm + a.tail_cost - 1) / a.tail_cost;
        c1 = static_cast<int>(cc < sc.tail_chunks ? cc : sc.tail_chunks);
      }
      const int slot = a.slot_ids ? a.slot_ids[b] : b;
      const bool slot_ok = slot >= 0 && slot < a.max_slots;
      const bool table_ok = static_cast<long long>(a.bt_stride) * kP >= T;
      // the segment's independent global reads are issued together: the cache's
      // length, the queries (tensor-core path) and the block-table entries
      // (through L2: a decode step wrote the lengths earlier in this launch)
      const int lens_v = slot_ok ? __ldcg(a.lens + slot * a.H + h) : 0;
      float fp8_ks = 1.0f, fp8_vs = 1.0f;   // FP8 pages: the head's key and value scales
      if constexpr (BITS == 8) {
        fp8_ks = a.fp8_scale[h];
        fp8_vs = a.fp8_scale[a.H + h];
      }
      const uint16_t* qrow = a.q + (static_cast<long long>(b) * a.Hq + h * a.g) * kD;
      uint4 qraw[4];   // tensor-core path: this lane's query words, q[gi][32 ti .. 32 ti + 31]
      if constexpr (IMPL != 1) {
        // variant 3 (GQA groups of at most 4): lanes of columns 4..7 hold heads 0..3 again
        const int gi = IMPL == 3 ? (lane >> 2) & 3 : lane >> 2, ti = lane & 3;
  #pragma unroll
        for (int i = 0; i < 4; ++i) qraw[i] = make_uint4(0u, 0u, 0u, 0u);
        if (gi < a.g && slot_ok && T > 0) {
          const uint4* src = reinterpret_cast<const uint4*>(qrow + gi * kD + 32 * ti);
  #pragma unroll
          for (int i = 0; i < 4; ++i) qraw[i] = src[i];
        }
      }
      Seg sg;
      sg.pages = a.pages;
      sg.bt = a.block_table + static_cast<long long>(b) * a.bt_stride;
      sg.kring = reinterpret_cast<const uint16_t*>(a.kring) + (slot_ok ? slot : 0) * a.kring_slot + h * a.kring_head;
      sg.vring = reinterpret_cast<const uint16_t*>(a.vring) + (slot_ok ? slot : 0) * a.vring_slot + h * a.vring_head;
      sg.H = a.H;
      sg.h = h;
      sg.T = T;
      sg.Tk = T & ~(kG - 1);
      sg.Tv = max(0, T - a.R);
      sg.R = a.R;
      sg.dtype = a.dtype;
      bool valid = slot_ok && T > 0;
      bool bad = false;
      if (valid && table_ok && (u1 > u0 || c1 > c0)) {
        // every page this warp will read must be inside the pool
        const int p_lo = u1 > u0 ? 2 * u0 : 2 * (nm + c0);
        const int p_hi = min(c1 > c0 ? 2 * (nm + c1) : 2 * u1, (T + kP - 1) / kP);
        for (int base = p_lo; base < p_hi; base += 32 * 8) {   // eight loads in flight per lane
          int pp[8];
  #pragma unroll
          for (int k = 0; k < 8; ++k) {
            const int lp = base + 32 * k + lane;
            pp[k] = lp < p_hi ? sg.bt[lp] : 0;
          }
  #pragma unroll
          for (int k = 0; k < 8; ++k) {
            if (base + 32 * k + lane < p_hi && (pp[k] < 0 || pp[k] >= a.num_pages)) {
              bad = true;
              report(a.status, S4KV_ERR_DEVICE, S4KV_DEV_BAD_PAGE, pp[k]);
            }
          }
        }
      }
      if (!slot_ok) {
        if (lane == 0) report(a.status, S4KV_ERR_DEVICE, S4KV_DEV_BAD_SLOT, slot);
      } else if (lens_v != T || T > a.max_seq_len) {
        valid = false;
        if (lane == 0) report(a.status, S4KV_ERR_DEVICE, S4KV_DEV_BAD_LENGTH, b);
      } else if (!table_ok) {
        valid = false;
        if (lane == 0) report(a.status, S4KV_ERR_DEVICE, S4KV_DEV_BAD_TABLE, b);
      }
      valid = valid && !__any_sync(0xffffffffu, bad) && !aborted;
      GenState gs;
      if (valid) {
        const int n = u1 - u0;
        float qv[32];   // tensor-core path: q[gi][32 ti + x], fp32
        if constexpr (IMPL != 1) {
  #pragma unroll
          for (int i = 0; i < 4; ++i) {   // heads >= g hold zero words, which widen to 0.0f
            const uint32_t w[4] = {qraw[i].x, qraw[i].y, qraw[i].z, qraw[i].w};
  #pragma unroll
            for (int j = 0; j < 4; ++j) {
              qv[8 * i + 2 * j] = widen16(static_cast<uint16_t>(w[j] & 0xffff), a.dtype);
              qv[8 * i + 2 * j + 1] = widen16(static_cast<uint16_t>(w[j] >> 16), a.dtype);
            }
          }
          MmaState ms;
          mma_init(ms);
          S4KV_TRACE(tr[7] += n; tlap(2); wslot = 12;)
          bool ok = true;
          if constexpr (BITS == 8) {
            // pages pg0 .. pg1 - 1 of the slice (the last unit may hold one page, or a partial one)
            const int pg0 = 2 * u0, pg1 = min(2 * u1, (T + kP - 1) / kP), np = pg1 - pg0;
            uint32_t qa[8][2];   // A operand, row gi: head gi's query in f16, channels c_0 c_1 | c_2 c_3 of slice kk
  #pragma unroll
            for (int kk = 0; kk < 8; ++kk) {
              qa[kk][0] = pack_f16x2(qv[4 * kk], qv[4 * kk + 1]);
              qa[kk][1] = pack_f16x2(qv[4 * kk + 2], qv[4 * kk + 3]);
            }
            const float zscale = a.sm_scale_log2 * fp8_ks;
            uint8_t* region = sm.region[warp];
            // pool pages pg0 + 32 k + lane, held one batch of 32 ahead of the copies
            auto page_of = [&](int k) {
              const int lp = pg0 + 32 * k + lane;
              return lp < pg1 ? sg.bt[lp] : 0;
            };
            int curp = page_of(0), nxtp = page_of(1), cur_k = 0;
            auto issue_page = [&](int st, int i) {   // i = 0, 1, 2, ... in order
              if ((i >> 5) != cur_k) {
                curp = nxtp;
                ++cur_k;
                nxtp = page_of(cur_k + 1);
              }
              const int pp = __shfl_sync(0xffffffffu, curp, i & 31);
              fence_proxy_async();   // earlier generic reads of the stage come first
              __syncwarp();
              if (lane == 0) {
                mbar_expect_tx(&bar[st], Rec<8>::kBytes);
                bulk_load_hint(region + st * Rec<8>::kBytes, rec_at<8>(sg, pp), Rec<8>::kBytes, &bar[st], once);
              }
              pend |= 1u << st;
            };
            for (int i = 0; i < np && i < kFp8Stages; ++i) issue_page(i, i);
            float m = -INFINITY, l = 0.0f;
            int st = 0;
            for (int i = 0; i < np; ++i) {
              if (!wait(st)) {
                ok = false;
                break;
              }
              const char* rec = reinterpret_cast<const char*>(region + st * Rec<8>::kBytes);
              const int nvalid = T - kP * (pg0 + i);
              if (nvalid < kP) fp8_page<true>(rec, ms, m, l, qa, zscale, nvalid);
              else fp8_page<false>(rec, ms, m, l, qa, zscale, kP);
              if (i + kFp8Stages < np) issue_page(st, i + kFp8Stages);
              st = st + 1 == kFp8Stages ? 0 : st + 1;
            }
            // into the MMA state's form (heads 2ti, 2ti + 1 per lane; sums in lanes gi = 0)
            l += __shfl_xor_sync(0xffffffffu, l, 1);
            l += __shfl_xor_sync(0xffffffffu, l, 2);
            const int ti = lane & 3;
            ms.m0 = __shfl_sync(0xffffffffu, m, 8 * ti);
            ms.m1 = __shfl_sync(0xffffffffu, m, 8 * ti + 4);
            const float l0 = __shfl_sync(0xffffffffu, l, 8 * ti), l1 = __shfl_sync(0xffffffffu, l, 8 * ti + 4);
            ms.l0 = lane < 4 ? l0 : 0.0f;
            ms.l1 = lane < 4 ? l1 : 0.0f;
  #pragma unroll
            for (int mt = 0; mt < 8; ++mt)
  #pragma unroll
              for (int e = 0; e < 4; ++e) ms.o[mt][e] *= fp8_vs;
            S4KV_TRACE(tlap(3);)
          } else {
            // Pool pages of main groups u0 + 32 k + lane (two per group), held in
            // registers one batch of 32 groups ahead of the copies that need them.
            auto load_batch = [&](int k, int& x0, int& x1) {
              const int jj = u0 + 32 * k + lane;
              x0 = x1 = 0;
              if (jj < u1) {
                x0 = sg.bt[2 * jj];
                x1 = sg.bt[2 * jj + 1];
              }
            };
            int cur0, cur1, nxt0, nxt1, cur_k = 0;
            load_batch(0, cur0, cur1);
            load_batch(1, nxt0, nxt1);
            auto issue_group = [&](int s, int j) {   // j = 0, 1, 2, ... in order
              if ((j >> 5) != cur_k) {
                cur0 = nxt0;
                cur1 = nxt1;
                ++cur_k;
                load_batch(cur_k + 1, nxt0, nxt1);
              }
              const int p0 = __shfl_sync(0xffffffffu, cur0, j & 31);
              const int p1 = __shfl_sync(0xffffffffu, cur1, j & 31);
              issue_pp(s, p0, p1, sg);
            };
            for (int j = 0; j < n && j < kStages; ++j) issue_group(j, j);
            for (int j = 0; j < n; ++j) {
              const int s = j & 1;
              if (!wait(s)) { ok = false; break; }
              mma_group<IMPL >= 2, BITS, IMPL == 3>(reinterpret_cast<const char*>(s ? st1 : st0), ms, ptile, qv,
                                         a.sm_scale_log2, kLoAbove / a.sm_scale_log2);
              if (j + kStages < n) issue_group(s, j + kStages);
            }
            mma_unscale<BITS>(ms);
            S4KV_TRACE(tlap(3);)
            unsigned long long* ttail = nullptr;   // tail phase counters (tracing builds)
            // pool pages of the first 16 tail groups: lane i holds logical page 2 (nm + c0) + i
            int tpg = 0;
            {
              const int lp = 2 * (nm + c0) + lane;
              if (c1 > c0 && lp < min(2 * (nm + c1), (T + kP - 1) / kP)) tpg = sg.bt[lp];
            }
            S4KV_TRACE(ttail = tr + 8; wslot = 13;)
            // Tail groups, one batch of bulk copies each into the warp's region: the
            // page records (keys and, where values are quantized, values) or the
            // key-ring rows, then the value-ring rows, one copy per row by the row's lane.
            for (int c = c0; ok && c < c1; ++c) {
              const int grp = nm + c;
              const int t0 = 32 * grp, t1 = min(t0 + kG, T);
              const bool kquant = t0 + kG <= sg.Tk;
              const bool vrec = t0 < sg.Tv;
              const bool kring_staged = !kquant && !vrec && t1 - t0 <= kKringStageMax;
              const int np = (t0 + kP < T) ? 2 : 1;
              const int vt0 = max(t0, sg.Tv);
              const int nv = max(0, t1 - vt0);
              const int voff = kring_staged ? (t1 - t0) * kD * 2 : kVoffRecsB<BITS>;
              uint32_t bytes = nv * kD * 2;
              if (vrec) bytes += np * F::kBytes;
              else if (kquant) bytes += np * (F::kKm + 512);
              if (kring_staged) bytes += (t1 - t0) * kD * 2;
              const int tp0 = __shfl_sync(0xffffffffu, tpg, (2 * (c - c0)) & 31);
              const int tp1 = __shfl_sync(0xffffffffu, tpg, (2 * (c - c0) + 1) & 31);
              fence_proxy_async();   // earlier generic accesses of the region come first
              __syncwarp();
              if (lane == 0) {
                mbar_expect_tx(&bar[0], bytes);
                if (vrec || kquant) {
                  const bool held = c - c0 < 16;
                  const char* r0 = held ? rec_at<BITS>(sg, tp0) : rec_of<BITS>(sg, 2 * grp);
                  const char* r1 = np < 2 ? r0 : held ? rec_at<BITS>(sg, tp1) : rec_of<BITS>(sg, 2 * grp + 1);
                  // whole records, or only the key codes and key metadata when no value is quantized
                  const uint32_t rb = vrec ? F::kBytes : F::kKm + 512;
                  bulk_load_hint(st0, r0, rb, &bar[0], once);
                  if (np == 2) bulk_load_hint(st0 + RS, r1, rb, &bar[0], once);
                }
                if (kring_staged) bulk_load_hint(st0, sg.kring, (t1 - t0) * kD * 2, &bar[0], once);
              }
              __syncwarp();
              if (lane < nv) {
                const int t = vt0 + lane;
                bulk_load_hint(st0 + voff + (t - t0) * kVRow, sg.vring + static_cast<long long>(t % sg.R) * kD, kD * 2,
                               &bar[0], once);
              }
              pend |= 1u;
              if (!wait(0)) {
                ok = false;
                break;
              }
              tail_group<BITS>(sg, grp, ms, ptile, qv, reinterpret_cast<const char*>(st0),
                         kring_staged ? reinterpret_cast<const uint16_t*>(st0) : sg.kring,
                         reinterpret_cast<const char*>(st0 + voff), zero_s, a.sm_scale_log2, T, T, ttail);
              S4KV_TRACE(tr[11] += 1;)
            }
          }
          if (ok) mma_to_gen(ms, gs, reinterpret_cast<float*>(st0));
          else {
            fail(b);
            gen_init(gs);
          }
          S4KV_TRACE(tlap(4);)
        } else {
          gen_init(gs);
          // query block for the FFMA path: lane l writes channels 4l..4l+3
          for (int j = 0; j < kNH; ++j) {
            float v[4] = {0.0f, 0.0f, 0.0f, 0.0f};
            if (j < a.g) ring_quad(qrow + j * kD, lane, a.dtype, v);
            *reinterpret_cast<float4*>(q_s + j * kD + 4 * lane) = make_float4(v[0], v[1], v[2], v[3]);
          }
          __syncwarp();
          for (int j = 0; j < n && j < kStages; ++j) issue(j, 2 * (u0 + j), 2, sg);
          for (int j = 0; j < n; ++j) {
            const int s = j & 1;
            if (!wait(s)) {
              fail(b);
              gen_init(gs);
              break;
            }
            ffma_group(reinterpret_cast<const char*>(s ? st1 : st0), gs, ptile, qp, q_s, a.sm_scale_log2);
            if (j + kStages < n) issue(s, 2 * (u0 + j + kStages), 2, sg);
          }
        }
        if constexpr (IMPL == 1) {
          // tail chunks: page records (when any of their keys or values are
          // quantized) staged in stage 0
          for (int c = c0; c < c1 && !aborted; ++c) {
            const int grp = nm + c;
            const int np = (32 * grp + kP < T) ? 2 : 1;
            issue(0, 2 * grp, np, sg);
            if (!wait(0)) {
              fail(b);
              gen_init(gs);
              break;
            }
            tail_chunk(sg, grp, gs, ptile, q_s, reinterpret_cast<const char*>(st0), a.sm_scale_log2);
          }
        }
      } else {
        gen_init(gs);
      }

      // ---- output, or the partial that merge_kernel combines ----
      if (seg_start >= r0 && lane == 0) {   // this warp holds the segment's first unit: its merge descriptor
        int ncon = 0;
        if (!own && slot_ok) ncon = owner_of(seg_end - 1, C, n_act) - gw + 1;
        const long long first = 2LL * gw + (seg_start <= r0 ? 0 : 1);
        meta_of(a)[static_cast<long long>(b) * a.H + h] =
            static_cast<long long>(static_cast<unsigned>(first)) | (static_cast<long long>(ncon) << 32);
      }
      if (own || !slot_ok) {
  #pragma unroll
        for (int j = 0; j < kNH; ++j) {
          if (j < a.g) {
            const float inv = gs.l[j] > 0.0f ? 1.0f / gs.l[j] : 0.0f;
            store_out(a, static_cast<long long>(b) * a.Hq + h * a.g + j, lane,
                      make_float4(gs.o[j][0] * inv, gs.o[j][1] * inv, gs.o[j][2] * inv, gs.o[j][3] * inv));
          }
        }
      } else {
        S4KV_TRACE(const unsigned long long tf0 = global_ns();)
        const int k = seg_start <= r0 ? 0 : 1;
        const long long part_floats = partial_floats(a.pcols);
        float* P = a.ws + (2LL * gw + k) * part_floats;
  #pragma unroll
        for (int j = 0; j < kNH; ++j) {
          if (j < a.g) {
            *reinterpret_cast<float4*>(P + j * kD + 4 * lane) =
                make_float4(gs.o[j][0], gs.o[j][1], gs.o[j][2], gs.o[j][3]);
            if (lane == 0) {
              P[a.pcols * kD + 2 * j] = gs.m[j];
              P[a.pcols * kD + 2 * j + 1] = gs.l[j];
            }
          }
        }
        S4KV_TRACE(tr[14] += global_ns() - tf0;)
      }

      S4KV_TRACE(tlap(5);)
      // next segment
      seg_start = seg_end;
      if (++h == a.H) {
        h = 0;
        if (++b >= a.B) break;
        sc = seg_cost<BITS>(a.seq_lens[b], a.R, a.tail_cost);
      }
    }
    if (pend) fail(-1);   // never expected: every issued copy is waited for
    S4KV_TRACE({
      tr[1] = global_ns();
      if (lane == 0) {
        unsigned long long* out = reinterpret_cast<unsigned long long*>(meta_of(a) + meta_words(a.B, a.H)) +
                                  static_cast<long long>(gw) * kTraceWords;
        for (int i = 0; i < kTraceWords; ++i) out[i] = tr[i];
      }
    })
  }
  // decode step: the combine of split segments, in the same launch
  if constexpr (STEP && kStepMerge) {
    grid_sync(a);
    unsigned long long t_seg = 0, t_ld = 0;
    merge_items(a, static_cast<long long>(blockIdx.x) * kWarps + warp, static_cast<long long>(gridDim.x) * kWarps,
                t_seg, t_ld);
  }
}

// ---- merge of split segments ---------------------------------------------------------
// Launched right behind decode_kernel (programmatic dependent launch): it waits
// for the attention grid to complete, then merges (see merge_items).
__global__ void __launch_bounds__(32 * kMergeWarps) merge_kernel(DecodeArgs a) {
  S4KV_TRACE(const unsigned long long tm_start = global_ns();)
  asm volatile("griddepcontrol.wait;" ::: "memory");   // decode_kernel has completed; its writes are visible
  S4KV_TRACE(const unsigned long long tm_go = global_ns();)
  unsigned long long tm_seg = 0, tm_ld = 0;   // (tracing builds)
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  (void)lane;
  merge_items(a, static_cast<long long>(blockIdx.x) * kMergeWarps + warp,
              static_cast<long long>(gridDim.x) * kMergeWarps, tm_seg, tm_ld);
  S4KV_TRACE({
    // after the decode warps' words: (wait released, descriptor read, loads landed, end) of merge warp i
    const long long mw = static_cast<long long>(blockIdx.x) * kMergeWarps + warp;
    if (lane == 0 && mw < a.grid_warps) {
      unsigned long long* out = reinterpret_cast<unsigned long long*>(meta_of(a) + meta_words(a.B, a.H)) +
                                static_cast<long long>(a.grid_warps) * kTraceWords + 4 * mw;
      out[0] = tm_go;
      out[1] = tm_seg;
      out[2] = tm_ld;
      out[3] = global_ns();
    }
    (void)tm_start;
  })
}

}  // namespace

size_t decode_meta_bytes(int B, int H) { return static_cast<size_t>(meta_words(B, H)) * sizeof(long long); }

int decode_threads(int impl) { return 32 * (impl == 1 ? warps_of<1>() : warps_of<0>()); }
int decode_warps_per_cta(int impl) { return impl == 1 ? warps_of<1>() : warps_of<0>(); }
size_t decode_partial_bytes(int g) { return static_cast<size_t>(partial_floats(g)) * sizeof(float); }
size_t decode_trace_bytes_per_warp() { return kTraceWords ? static_cast<size_t>(kTraceWords + 4) * 8 : 0; }

size_t decode_smem_bytes(int impl, int B) {
  const size_t base = impl == 1 ? prefix_offset<1>() : prefix_offset<0>();
  return base + static_cast<size_t>(B + 1) * sizeof(long long);
}

namespace {
template <int IMPL, int BITS, bool STEP = false>
cudaError_t prepare(int B, int* per_sm) {
  static size_t attr_bytes = 0;   // largest dynamic shared memory granted so far
  const size_t need = decode_smem_bytes(IMPL, B);
  const cudaError_t e = grant_smem(decode_kernel<IMPL, BITS, STEP>, need, &attr_bytes);
  if (e != cudaSuccess) return e;
  if (per_sm)
    return cudaOccupancyMaxActiveBlocksPerMultiprocessor(per_sm, decode_kernel<IMPL, BITS, STEP>,
                                                         32 * warps_of<IMPL>(), need);
  return cudaSuccess;
}

// The instantiations: tensor-core path (0), FFMA path (1, 4-bit only), tensor-core
// path with the key split (2), the split packed into one MMA for GQA groups of at
// most 4 heads (3), each for 4-bit and 2-bit records; the tensor-core path for FP8
// records.
cudaError_t prepare_any(int impl, int bits, int B, int* per_sm) {
  if (bits == 8) return prepare<0, 8>(B, per_sm);
  if (bits == 2)
    return impl == 3 ? prepare<3, 2>(B, per_sm) : impl == 2 ? prepare<2, 2>(B, per_sm) : prepare<0, 2>(B, per_sm);
  return impl == 1   ? prepare<1, 4>(B, per_sm)
         : impl == 2 ? prepare<2, 4>(B, per_sm)
         : impl == 3 ? prepare<3, 4>(B, per_sm)
                     : prepare<0, 4>(B, per_sm);
}
}  // namespace

int decode_ctas_per_sm(int impl, int B) {
  int n = 0;
  const cudaError_t e = prepare_any(impl, 4, B, &n);
  return e == cudaSuccess ? n : 0;
}

cudaError_t launch_decode_step(const DecodeArgs& a, int impl, int grid, cudaStream_t st) {
  const size_t smem = decode_smem_bytes(impl, a.B);
  if (impl == 1) return cudaErrorInvalidValue;   // the step runs on the tensor-core paths
  if (impl == 3 && a.g > 4) return cudaErrorInvalidValue;   // the packed split holds 4 heads
  int per_sm = 0;
  cudaError_t e;
  void (*kern)(DecodeArgs);
  if (a.bits == 8) {
    e = prepare<0, 8, true>(a.B, &per_sm);
    kern = decode_kernel<0, 8, true>;
  } else if (a.bits == 2) {
    e = impl == 3   ? prepare<3, 2, true>(a.B, &per_sm)
        : impl == 2 ? prepare<2, 2, true>(a.B, &per_sm)
                    : prepare<0, 2, true>(a.B, &per_sm);
    kern = impl == 3 ? decode_kernel<3, 2, true> : impl == 2 ? decode_kernel<2, 2, true> : decode_kernel<0, 2, true>;
  } else {
    e = impl == 3   ? prepare<3, 4, true>(a.B, &per_sm)
        : impl == 2 ? prepare<2, 4, true>(a.B, &per_sm)
                    : prepare<0, 4, true>(a.B, &per_sm);
    kern = impl == 3 ? decode_kernel<3, 4, true> : impl == 2 ? decode_kernel<2, 4, true> : decode_kernel<0, 4, true>;
  }
  if (e != cudaSuccess) return e;
  if (per_sm <= 0 || grid % per_sm != 0) return cudaErrorCooperativeLaunchTooLarge;   // every CTA resident
  // every CTA must be resident at once for the grid barrier: a cooperative launch
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>(grid));
  cfg.blockDim = dim3(32 * warps_of<0>());
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeCooperative;
  attr[0].val.cooperative = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  e = cudaLaunchKernelEx(&cfg, kern, a);
  if (e != cudaSuccess || kStepMerge) return e;   // with kStepMerge the merge ran inside
  return launch_merge(merge_kernel, a, static_cast<long long>(a.B) * a.H * a.g, grid, st);
}

cudaError_t launch_decode(const DecodeArgs& a, int impl, int grid, cudaStream_t st) {
  const size_t smem = decode_smem_bytes(impl, a.B);
  if (a.bits != 4 && impl == 1) return cudaErrorInvalidValue;   // FFMA path: 4-bit records only
  if (a.bits == 8 && impl != 0) return cudaErrorInvalidValue;
  if (impl == 3 && a.g > 4) return cudaErrorInvalidValue;   // the packed split holds 4 heads
  cudaError_t e = prepare_any(impl, a.bits, a.B, nullptr);
  if (e != cudaSuccess) return e;
  const int threads = 32 * (impl == 1 ? warps_of<1>() : warps_of<0>());
  if (a.bits == 8) {
    decode_kernel<0, 8><<<grid, threads, smem, st>>>(a);
  } else if (a.bits == 2) {
    if (impl == 3) decode_kernel<3, 2><<<grid, threads, smem, st>>>(a);
    else if (impl == 2) decode_kernel<2, 2><<<grid, threads, smem, st>>>(a);
    else decode_kernel<0, 2><<<grid, threads, smem, st>>>(a);
  } else {
    if (impl == 1) decode_kernel<1, 4><<<grid, threads, smem, st>>>(a);
    else if (impl == 2) decode_kernel<2, 4><<<grid, threads, smem, st>>>(a);
    else if (impl == 3) decode_kernel<3, 4><<<grid, threads, smem, st>>>(a);
    else decode_kernel<0, 4><<<grid, threads, smem, st>>>(a);
  }
  e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  // merge_kernel right behind it, launched programmatically: its blocks may be
  // scheduled while decode_kernel drains and wait for its completion on the device
  return launch_merge(merge_kernel, a, static_cast<long long>(a.B) * a.H * a.g, grid, st);
}

}  // namespace s4kv
