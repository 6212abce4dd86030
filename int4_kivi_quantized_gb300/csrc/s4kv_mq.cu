// Multi-query attention: causal attention of the last nq tokens of every
// sequence over the cache after they were appended ("给 KV cache 减肥" section 2:
// P = softmax(QK^T / sqrt d), output P V; "4.4 KV Cache 量化" section 3.2: the
// residual and the quantized history take part together). Four kernels share the
// decode path's cost line, staging and merge workspace:
//  * mq_kernel: KIVI pages, the scales folded into every warp's 8 columns;
//  * mqd_kernel: KIVI pages, each key group restored once per team for mma.sync
//    on 16 columns a warp (wide calls);
//  * mqt_kernel: the same restored groups fed to tcgen05, accumulators in tensor
//    memory, warp-specialized (from S4KV_MQ_TC_MIN_COLS columns, or chosen);
//  * mq_fp8_kernel: FP8 pages, 16 columns a warp; wide calls on FP8 pages take
//    mqt_kernel<8>, which widens each group's codes once for tcgen05.
// mq_merge_kernel combines split segments' partials.

#include "s4kv_kernels.cuh"

// Multi-query over KIVI pages: the column count (nq g) from which each key group is
// restored once per team rather than folded into every warp's columns (measured on
// Llama-3.1-8B shapes: folding is 1.75x faster at 32 columns, restoring 1.2x at 64).
#ifndef S4KV_MQ_RESTORE_MIN_COLS
#define S4KV_MQ_RESTORE_MIN_COLS 64
#endif
// ... and from which the restored group feeds tcgen05 (mqt_kernel) instead, on both
// page formats: past 48 columns a team of the mma.sync kernels needs 7 or more of a
// CTA's 12 warps, so a CTA holds one team. Measured (GB/s; folding or FP8 mma.sync
// against tcgen05): KIVI pages on Llama-3.1-8B shapes 963 / 858 at 40 columns,
// 953 / 860 at 48, 611 / 859 at 56; Qwen2.5-7B shapes at 49 columns 635 / 973. FP8
// pages: 2171 / 1170 at 32 and 1596 / 1207 at 48 columns (Llama-3.1-8B shapes), 1282 /
// 1504 at 49 and 936 / 1169 at 70 (Qwen2.5-7B shapes), 1180 / 1204 at 64. The mma.sync
// restore kernel is then taken only when chosen.
#ifndef S4KV_MQ_TC_MIN_COLS_KIVI
#define S4KV_MQ_TC_MIN_COLS_KIVI 49
#endif
#ifndef S4KV_MQ_TC_MIN_COLS
#define S4KV_MQ_TC_MIN_COLS 49
#endif

namespace s4kv {
namespace {

// ---- multi-query attention: a chunk of query tokens per sequence ------------------------
// Causal attention of the last nq <= 16 tokens of every sequence (a chunk of a
// chunked prefill, or the tokens a speculative step verifies) over the length-T
// state after the chunk was appended: query i, at position T - nq + i, sees
// tokens 0 .. T - nq + i. Column c = i * g + j pairs query token i with head j
// of the kv head. A team of tw = ceil(nq g / 8) warps works on one slice of the
// cost line: its leader stages each key group once for the whole team (full
// barriers), every warp runs the decode arithmetic on its own 8 columns and
// then marks the stage free (empty barriers, one arrival per warp). Main groups
// need no mask (nq <= R puts them below every column's limit); tail groups
// take each column's limit.
template <int BITS>
__global__ void __launch_bounds__(32 * S4KV_DECODE_WARPS, S4KV_DECODE_MIN_CTAS) mq_kernel(DecodeArgs a) {
  using F = Rec<BITS>;
  constexpr int RS = kRecStrideB<BITS>;
  constexpr int kWarps = S4KV_DECODE_WARPS;
  constexpr int kThreads = 32 * kWarps;
  using SmemT = Smem<kWarps>;
  extern __shared__ __align__(128) uint8_t smem_raw[];
  SmemT& sm = *reinterpret_cast<SmemT*>(smem_raw);
  long long* pre = reinterpret_cast<long long*>(smem_raw + prefix_offset<0>());   // [B + 1]
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int tw = a.tw, tpc = kWarps / tw;
  const int team = warp / tw, tile = warp - team * tw;
  const bool in_team = team < tpc;
  const int lead = in_team ? team * tw : warp;
  const bool leader = in_team && tile == 0;
  uint8_t* st0 = sm.region[lead];
  uint8_t* st1 = st0 + kStageBytesB<BITS>;
  uint64_t* full = sm.bar[lead];
  uint64_t* empty = sm.bar[lead] + kStages;
  float* ptile = sm.ptile[warp];
  // mma_to_gen scratch: a warp's own region (the leader's only once its team is done with it)
  float* scratch = reinterpret_cast<float*>(sm.region[warp]);

  if (leader && lane == 0) {
    mbar_init(&full[0], 1);
    mbar_init(&full[1], 1);
    mbar_init(&empty[0], tw);
    mbar_init(&empty[1], tw);
  }
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  __shared__ __align__(16) uint4 zero16;
  if (tid == 0) zero16 = make_uint4(0u, 0u, 0u, 0u);
  const uint32_t zero_s = smem_u32(&zero16);
  {
    long long carry = 0;
    __shared__ long long wt[kWarps];
    for (int base = 0; base < a.B; base += kThreads) {
      const int b = base + tid;
      const long long cnt = b < a.B ? a.H * seg_cost(a.seq_lens[b], a.R, a.tail_cost).cost : 0;
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
  int n_act = static_cast<int>(gridDim.x) * tpc;
  if (a.max_warps > 0 && a.max_warps < n_act) n_act = a.max_warps;   // the option caps teams here
  {
    const long long cap = (C + kMinUnits - 1) / kMinUnits;
    if (cap < n_act) n_act = static_cast<int>(cap);
  }
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  if (!in_team) return;
  const int gteam = blockIdx.x * tpc + team;
  if (gteam >= n_act) return;
  const int gw = blockIdx.x * kWarps + warp;
  const long long r0 = gteam * C / n_act, r1 = (gteam + 1) * C / n_act;
  const uint64_t once = policy_evict_first();
  const int cols = a.nq * a.g;

  uint32_t fph = 0, eph = 0, epend = 0, pend = 0;
  bool aborted = false;
  auto wait_full = [&](int s) -> bool {
    if (!mbar_wait(&full[s], (fph >> s) & 1u, aborted ? 0 : a.wait_ns)) return false;
    fph ^= 1u << s;
    pend &= ~(1u << s);
    return true;
  };
  auto release = [&](int s) {   // this warp is done reading stage s
    __syncwarp();
    if (lane == 0) asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(&empty[s])) : "memory");
    epend |= 1u << s;
  };
  auto claim = [&](int s) -> bool {   // leader: every warp of the team is done with stage s
    if (!((epend >> s) & 1u)) return true;
    if (!mbar_wait(&empty[s], (eph >> s) & 1u, aborted ? 0 : a.wait_ns)) return false;
    eph ^= 1u << s;
    epend &= ~(1u << s);
    return true;
  };
  auto fail = [&](long long where) {
    if (lane == 0) report(a.status, S4KV_ERR_DEVICE_TIMEOUT, S4KV_DEV_TIMEOUT, static_cast<int>(where));
    aborted = true;
    for (int s = 0; s < kStages; ++s) {
      if ((pend >> s) & 1u) {
        mbar_wait(&full[s], (fph >> s) & 1u, kDrainNs);
        fph ^= 1u << s;
        pend &= ~(1u << s);
      }
    }
  };

  int b;
  {
    int lo = 0, hi = a.B - 1;
    while (lo < hi) {
      const int mid = (lo + hi + 1) >> 1;
      if (pre[mid] <= r0) lo = mid; else hi = mid - 1;
    }
    b = lo;
  }
  SegCost sc = seg_cost(a.seq_lens[b], a.R, a.tail_cost);
  int h = static_cast<int>((r0 - pre[b]) / sc.cost);
  long long seg_start = pre[b] + h * sc.cost;

  while (seg_start < r1) {
    const long long seg_end = seg_start + sc.cost;
    const int T = max(a.seq_lens[b], 0);
    const long long lo = max(r0, seg_start) - seg_start, hi = min(r1, seg_end) - seg_start;
    const bool own = lo == 0 && hi == sc.cost;
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
    const int lens_v = slot_ok ? a.lens[slot * a.H + h] : 0;
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
      const int p_lo = u1 > u0 ? 2 * u0 : 2 * (nm + c0);
      const int p_hi = min(c1 > c0 ? 2 * (nm + c1) : 2 * u1, (T + kP - 1) / kP);
      for (int base = p_lo; base < p_hi; base += 32 * 8) {
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
    } else if (lens_v != T || T > a.max_seq_len || T < a.nq) {
      valid = false;
      if (lane == 0) report(a.status, S4KV_ERR_DEVICE, S4KV_DEV_BAD_LENGTH, b);
    } else if (!table_ok) {
      valid = false;
      if (lane == 0) report(a.status, S4KV_ERR_DEVICE, S4KV_DEV_BAD_TABLE, b);
    }
    valid = valid && !__any_sync(0xffffffffu, bad) && !aborted;
    // row of out / q for column c of this segment
    auto row_of = [&](int c) -> long long {
      return (static_cast<long long>(b) * a.nq + c / a.g) * a.Hq + h * a.g + c % a.g;
    };
    GenState gs;
    if (valid) {
      const int n = u1 - u0;
      const int gi = lane >> 2, ti = lane & 3;
      float qv[32];
      {
        const int c = 8 * tile + gi;
        uint4 qraw[4];
#pragma unroll
        for (int i = 0; i < 4; ++i) qraw[i] = make_uint4(0u, 0u, 0u, 0u);
        if (c < cols) {
          const uint4* src = reinterpret_cast<const uint4*>(a.q + row_of(c) * kD + 32 * ti);
#pragma unroll
          for (int i = 0; i < 4; ++i) qraw[i] = src[i];
        }
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          const uint32_t w[4] = {qraw[i].x, qraw[i].y, qraw[i].z, qraw[i].w};
#pragma unroll
          for (int j = 0; j < 4; ++j) {
            qv[8 * i + 2 * j] = widen16(static_cast<uint16_t>(w[j] & 0xffff), a.dtype);
            qv[8 * i + 2 * j + 1] = widen16(static_cast<uint16_t>(w[j] >> 16), a.dtype);
          }
        }
      }
      // causal limits of this lane's accumulator columns 2ti, 2ti+1 of the tile
      const int ca = 8 * tile + 2 * ti, cb = ca + 1;
      const int lim0 = ca < cols ? T - a.nq + ca / a.g + 1 : T;
      const int lim1 = cb < cols ? T - a.nq + cb / a.g + 1 : T;
      MmaState ms;
      mma_init(ms);
      // leader: pool pages of main groups u0 + 32 k + lane, a batch ahead
      int cur0 = 0, cur1 = 0, nxt0 = 0, nxt1 = 0, cur_k = 0;
      auto load_batch = [&](int k, int& x0, int& x1) {
        const int jj = u0 + 32 * k + lane;
        x0 = x1 = 0;
        if (jj < u1) {
          x0 = sg.bt[2 * jj];
          x1 = sg.bt[2 * jj + 1];
        }
      };
      auto issue_group = [&](int s, int j) {
        if ((j >> 5) != cur_k) {
          cur0 = nxt0;
          cur1 = nxt1;
          ++cur_k;
          load_batch(cur_k + 1, nxt0, nxt1);
        }
        const int p0 = __shfl_sync(0xffffffffu, cur0, j & 31);
        const int p1 = __shfl_sync(0xffffffffu, cur1, j & 31);
        fence_proxy_async();
        __syncwarp();
        if (lane == 0) {
          uint8_t* dst = s ? st1 : st0;
          mbar_expect_tx(&full[s], 2 * F::kBytes);
          bulk_load_hint(dst, rec_at<BITS>(sg, p0), F::kBytes, &full[s], once);
          bulk_load_hint(dst + RS, rec_at<BITS>(sg, p1), F::kBytes, &full[s], once);
        }
        pend |= 1u << s;
      };
      bool ok = true;
      if (leader) {
        load_batch(0, cur0, cur1);
        load_batch(1, nxt0, nxt1);
        for (int j = 0; j < n && j < kStages; ++j) {
          if (!claim(j)) { ok = false; break; }
          issue_group(j, j);
        }
      }
      for (int j = 0; ok && j < n; ++j) {
        const int s = j & 1;
        if (!wait_full(s)) { ok = false; break; }
        mma_group<true, BITS>(reinterpret_cast<const char*>(s ? st1 : st0), ms, ptile, qv, a.sm_scale_log2,
                              kLoAbove / a.sm_scale_log2);
        release(s);
        if (leader && j + kStages < n) {
          if (!claim(s)) { ok = false; break; }
          issue_group(s, j + kStages);
        }
      }
      mma_unscale<BITS>(ms);
      int tpg = 0;
      {
        const int lp = 2 * (nm + c0) + lane;
        if (c1 > c0 && lp < min(2 * (nm + c1), (T + kP - 1) / kP)) tpg = sg.bt[lp];
      }
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
        const int tp0 = __shfl_sync(0xffffffffu, tpg, (2 * (c - c0)) & 31);
        const int tp1 = __shfl_sync(0xffffffffu, tpg, (2 * (c - c0) + 1) & 31);
        if (leader) {
          // the batch overwrites the whole region: the team must be done with both stages
          if (!claim(0) || !claim(1)) { ok = false; break; }
          uint32_t bytes = nv * kD * 2;
          if (vrec) bytes += np * F::kBytes;
          else if (kquant) bytes += np * (F::kKm + 512);
          if (kring_staged) bytes += (t1 - t0) * kD * 2;
          fence_proxy_async();
          __syncwarp();
          if (lane == 0) {
            mbar_expect_tx(&full[0], bytes);
            if (vrec || kquant) {
              const bool held = c - c0 < 16;
              const char* ra = held ? rec_at<BITS>(sg, tp0) : rec_of<BITS>(sg, 2 * grp);
              const char* rb = np < 2 ? ra : held ? rec_at<BITS>(sg, tp1) : rec_of<BITS>(sg, 2 * grp + 1);
              const uint32_t nb = vrec ? F::kBytes : F::kKm + 512;
              bulk_load_hint(st0, ra, nb, &full[0], once);
              if (np == 2) bulk_load_hint(st0 + RS, rb, nb, &full[0], once);
            }
            if (kring_staged) bulk_load_hint(st0, sg.kring, (t1 - t0) * kD * 2, &full[0], once);
          }
          __syncwarp();
          if (lane < nv) {
            const int t = vt0 + lane;
            bulk_load_hint(st0 + voff + (t - t0) * kVRow, sg.vring + static_cast<long long>(t % sg.R) * kD, kD * 2,
                           &full[0], once);
          }
          pend |= 1u;
        }
        if (!wait_full(0)) { ok = false; break; }
        tail_group<BITS>(sg, grp, ms, ptile, qv, reinterpret_cast<const char*>(st0),
                   kring_staged ? reinterpret_cast<const uint16_t*>(st0) : sg.kring,
                   reinterpret_cast<const char*>(st0 + voff), zero_s, a.sm_scale_log2, lim0, lim1, nullptr);
        release(0);
      }
      if (ok && leader && (!claim(0) || !claim(1))) ok = false;   // scratch below is the staging region
      if (ok) mma_to_gen(ms, gs, scratch);
      else {
        fail(b);
        gen_init(gs);
      }
    } else {
      gen_init(gs);
    }

    // ---- output, or the partial that mq_merge_kernel combines ----
    if (leader && seg_start >= r0 && lane == 0) {
      int ncon = 0;
      if (!own && slot_ok) ncon = owner_of(seg_end - 1, C, n_act) - gteam + 1;
      const long long first = 2LL * gteam + (seg_start <= r0 ? 0 : 1);
      meta_of(a)[static_cast<long long>(b) * a.H + h] =
          static_cast<long long>(static_cast<unsigned>(first)) | (static_cast<long long>(ncon) << 32);
    }
    if (own || !slot_ok) {
#pragma unroll
      for (int j = 0; j < kNH; ++j) {
        const int c = 8 * tile + j;
        if (c < cols) {
          const float inv = gs.l[j] > 0.0f ? 1.0f / gs.l[j] : 0.0f;
          store_out(a, row_of(c), lane,
                    make_float4(gs.o[j][0] * inv, gs.o[j][1] * inv, gs.o[j][2] * inv, gs.o[j][3] * inv));
        }
      }
    } else {
      const int k = seg_start <= r0 ? 0 : 1;
      float* P = a.ws + (2LL * gw + k) * partial_floats(a.pcols);
#pragma unroll
      for (int j = 0; j < kNH; ++j) {
        *reinterpret_cast<float4*>(P + j * kD + 4 * lane) = make_float4(gs.o[j][0], gs.o[j][1], gs.o[j][2], gs.o[j][3]);
        if (lane == 0) {
          P[a.pcols * kD + 2 * j] = gs.m[j];
          P[a.pcols * kD + 2 * j + 1] = gs.l[j];
        }
      }
    }
    seg_start = seg_end;
    if (++h == a.H) {
      h = 0;
      if (++b >= a.B) break;
      sc = seg_cost(a.seq_lens[b], a.R, a.tail_cost);
    }
  }
  if (pend) fail(-1);
}

// Multi-query attention over FP8 pages: the same causal reading and cost line as
// mq_kernel (FP8 segments have no tail), with 16 columns per warp. A team of
// tw = ceil(nq g / 16) warps shares each page record: its leader stages single
// pages into a ring of 2 tw stages spread over the team's regions (full
// barriers), every warp runs fp8_page_mq on its 16 columns and then marks the
// stage free (empty barriers). Partials hold 16 columns (pcols = 16).
__global__ void __launch_bounds__(32 * S4KV_DECODE_WARPS, S4KV_DECODE_MIN_CTAS) mq_fp8_kernel(DecodeArgs a) {
  constexpr int kWarps = S4KV_DECODE_WARPS;
  constexpr int kThreads = 32 * kWarps;
  constexpr int RB = Rec<8>::kBytes;
  static_assert(2 * RB <= kRegion, "two FP8 stages fit a warp's region");
  using SmemT = Smem<kWarps>;
  extern __shared__ __align__(128) uint8_t smem_raw[];
  SmemT& sm = *reinterpret_cast<SmemT*>(smem_raw);
  long long* pre = reinterpret_cast<long long*>(smem_raw + prefix_offset<0>());   // [B + 1]
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int tw = a.tw, tpc = kWarps / tw;
  const int team = warp / tw, tile = warp - team * tw;
  const bool in_team = team < tpc;
  const int lead = in_team ? team * tw : warp;
  const bool leader = in_team && tile == 0;
  const int NS = 2 * tw;   // stage s: region of warp lead + s / 2, half s % 2
  auto stage = [&](int s) -> uint8_t* { return sm.region[lead + (s >> 1)] + (s & 1) * RB; };
  auto full_of = [&](int s) -> uint64_t* { return &sm.bar[lead + (s >> 1)][s & 1]; };
  auto empty_of = [&](int s) -> uint64_t* { return &sm.bar[lead + (s >> 1)][kStages + (s & 1)]; };
  float* scratch = reinterpret_cast<float*>(sm.region[warp]);   // mma_to_gen, once the team is done

  if (in_team && lane == 0) {
    mbar_init(&sm.bar[warp][0], 1);
    mbar_init(&sm.bar[warp][1], 1);
    mbar_init(&sm.bar[warp][kStages], tw);
    mbar_init(&sm.bar[warp][kStages + 1], tw);
  }
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  {
    long long carry = 0;
    __shared__ long long wt[kWarps];
    for (int base = 0; base < a.B; base += kThreads) {
      const int b = base + tid;
      const long long cnt = b < a.B ? a.H * seg_cost<8>(a.seq_lens[b], a.R, a.tail_cost).cost : 0;
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
  int n_act = static_cast<int>(gridDim.x) * tpc;
  if (a.max_warps > 0 && a.max_warps < n_act) n_act = a.max_warps;   // the option caps teams here
  {
    const long long cap = (C + kMinUnits - 1) / kMinUnits;
    if (cap < n_act) n_act = static_cast<int>(cap);
  }
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  if (!in_team) return;
  const int gteam = blockIdx.x * tpc + team;
  if (gteam >= n_act) return;
  const int gw = blockIdx.x * kWarps + warp;
  const long long r0 = gteam * C / n_act, r1 = (gteam + 1) * C / n_act;
  const uint64_t once = policy_evict_first();
  const int cols = a.nq * a.g;
  const int gi = lane >> 2, ti = lane & 3;
  auto team_sync = [&]() {   // named barrier of the team's warps (id 0 is __syncthreads)
    if (tw > 1) asm volatile("bar.sync %0, %1;" ::"r"(1 + team), "r"(32 * tw) : "memory");
    else __syncwarp();
  };

  uint32_t fph = 0, eph = 0, epend = 0, pend = 0;
  bool aborted = false;
  auto wait_full = [&](int s) -> bool {
    if (!mbar_wait(full_of(s), (fph >> s) & 1u, aborted ? 0 : a.wait_ns)) return false;
    fph ^= 1u << s;
    pend &= ~(1u << s);
    return true;
  };
  auto release = [&](int s) {   // this warp is done reading stage s
    __syncwarp();
    if (lane == 0) asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(empty_of(s))) : "memory");
    epend |= 1u << s;
  };
  auto claim = [&](int s) -> bool {   // leader: every warp of the team is done with stage s
    if (!((epend >> s) & 1u)) return true;
    if (!mbar_wait(empty_of(s), (eph >> s) & 1u, aborted ? 0 : a.wait_ns)) return false;
    eph ^= 1u << s;
    epend &= ~(1u << s);
    return true;
  };
  auto fail = [&](long long where) {
    if (lane == 0) report(a.status, S4KV_ERR_DEVICE_TIMEOUT, S4KV_DEV_TIMEOUT, static_cast<int>(where));
    aborted = true;
    for (int s = 0; s < NS; ++s) {
      if ((pend >> s) & 1u) {
        mbar_wait(full_of(s), (fph >> s) & 1u, kDrainNs);
        fph ^= 1u << s;
        pend &= ~(1u << s);
      }
    }
  };

  int b;
  {
    int lo = 0, hi = a.B - 1;
    while (lo < hi) {
      const int mid = (lo + hi + 1) >> 1;
      if (pre[mid] <= r0) lo = mid; else hi = mid - 1;
    }
    b = lo;
  }
  SegCost sc = seg_cost<8>(a.seq_lens[b], a.R, a.tail_cost);
  int h = static_cast<int>((r0 - pre[b]) / sc.cost);
  long long seg_start = pre[b] + h * sc.cost;

  while (seg_start < r1) {
    const long long seg_end = seg_start + sc.cost;
    const int T = max(a.seq_lens[b], 0);
    const long long lo = max(r0, seg_start) - seg_start, hi = min(r1, seg_end) - seg_start;
    const bool own = lo == 0 && hi == sc.cost;
    const int nm = sc.main_groups;
    const int u0 = static_cast<int>(lo < nm ? lo : nm), u1 = static_cast<int>(hi < nm ? hi : nm);
    const int slot = a.slot_ids ? a.slot_ids[b] : b;
    const bool slot_ok = slot >= 0 && slot < a.max_slots;
    const bool table_ok = static_cast<long long>(a.bt_stride) * kP >= T;
    const int lens_v = slot_ok ? a.lens[slot * a.H + h] : 0;
    const float ks = a.fp8_scale[h], vs = a.fp8_scale[a.H + h];
    Seg sg;
    sg.pages = a.pages;
    sg.bt = a.block_table + static_cast<long long>(b) * a.bt_stride;
    sg.H = a.H;
    sg.h = h;
    sg.T = T;
    const int npT = (T + kP - 1) / kP;
    const int pg0 = 2 * u0, pg1 = min(2 * u1, npT), np = max(0, pg1 - pg0);
    bool valid = slot_ok && T > 0;
    bool bad = false;
    if (valid && table_ok && np > 0) {
      for (int base = pg0; base < pg1; base += 32 * 8) {
        int pp[8];
#pragma unroll
        for (int k = 0; k < 8; ++k) {
          const int lp = base + 32 * k + lane;
          pp[k] = lp < pg1 ? sg.bt[lp] : 0;
        }
#pragma unroll
        for (int k = 0; k < 8; ++k) {
          if (base + 32 * k + lane < pg1 && (pp[k] < 0 || pp[k] >= a.num_pages)) {
            bad = true;
            report(a.status, S4KV_ERR_DEVICE, S4KV_DEV_BAD_PAGE, pp[k]);
          }
        }
      }
    }
    if (!slot_ok) {
      if (lane == 0) report(a.status, S4KV_ERR_DEVICE, S4KV_DEV_BAD_SLOT, slot);
    } else if (lens_v != T || T > a.max_seq_len || T < a.nq) {
      valid = false;
      if (lane == 0) report(a.status, S4KV_ERR_DEVICE, S4KV_DEV_BAD_LENGTH, b);
    } else if (!table_ok) {
      valid = false;
      if (lane == 0) report(a.status, S4KV_ERR_DEVICE, S4KV_DEV_BAD_TABLE, b);
    }
    valid = valid && !__any_sync(0xffffffffu, bad) && !aborted;
    auto row_of = [&](int c) -> long long {
      return (static_cast<long long>(b) * a.nq + c / a.g) * a.Hq + h * a.g + c % a.g;
    };
    float o[8][2][4];
#pragma unroll
    for (int mt = 0; mt < 8; ++mt)
#pragma unroll
      for (int ct = 0; ct < 2; ++ct)
#pragma unroll
        for (int e = 0; e < 4; ++e) o[mt][ct][e] = 0.0f;
    float m[2] = {-INFINITY, -INFINITY}, l[2] = {0.0f, 0.0f};
    bool ok = true;
    if (valid) {
      // A operand rows: columns c_lo = 16 tile + gi and c_hi = c_lo + 8 (zero past cols)
      const int c_lo = 16 * tile + gi, c_hi = c_lo + 8;
      uint32_t qa[8][4];
      {
        uint4 ql[4], qh[4];
#pragma unroll
        for (int i = 0; i < 4; ++i) ql[i] = qh[i] = make_uint4(0u, 0u, 0u, 0u);
        if (c_lo < cols) {
          const uint4* src = reinterpret_cast<const uint4*>(a.q + row_of(c_lo) * kD + 32 * ti);
#pragma unroll
          for (int i = 0; i < 4; ++i) ql[i] = src[i];
        }
        if (c_hi < cols) {
          const uint4* src = reinterpret_cast<const uint4*>(a.q + row_of(c_hi) * kD + 32 * ti);
#pragma unroll
          for (int i = 0; i < 4; ++i) qh[i] = src[i];
        }
        // channel 32 ti + 4 kk + j sits in word (kk / 2) of uint4 i = kk / 2 ... as 16-bit halves:
        // q words hold channels 32 ti + 2 w, + 1 (w = 0 .. 15)
        auto q2 = [&](const uint4 (&u)[4], int w) -> uint32_t {   // channels 32 ti + 2w, 2w + 1 as f16x2
          const uint4 x = u[w >> 2];
          const uint32_t r = (w & 3) == 0 ? x.x : (w & 3) == 1 ? x.y : (w & 3) == 2 ? x.z : x.w;
          if (a.dtype == S4KV_F16) return r;
          return pack_f16x2(widen16(static_cast<uint16_t>(r & 0xffff), S4KV_BF16),
                            widen16(static_cast<uint16_t>(r >> 16), S4KV_BF16));
        };
#pragma unroll
        for (int kk = 0; kk < 8; ++kk) {
          qa[kk][0] = q2(ql, 2 * kk);       // column c_lo, channels c_0, c_1
          qa[kk][1] = q2(qh, 2 * kk);       // column c_hi, c_0, c_1
          qa[kk][2] = q2(ql, 2 * kk + 1);   // column c_lo, c_2, c_3
          qa[kk][3] = q2(qh, 2 * kk + 1);
        }
      }
      // causal limits; pages wholly below every column's limit need no mask
      const int lim_lo = c_lo < cols ? T - a.nq + c_lo / a.g + 1 : T;
      const int lim_hi = c_hi < cols ? T - a.nq + c_hi / a.g + 1 : T;
      int free_end = min(lim_lo, lim_hi);
#pragma unroll
      for (int x = 1; x < 32; x <<= 1) free_end = min(free_end, __shfl_xor_sync(0xffffffffu, free_end, x));
      const float zscale = a.sm_scale_log2 * ks;
      // leader: pool pages pg0 + 32 k + lane, one batch of 32 ahead of the copies
      auto page_of = [&](int k) {
        const int lp = pg0 + 32 * k + lane;
        return lp < pg1 ? sg.bt[lp] : 0;
      };
      int curp = 0, nxtp = 0, cur_k = 0;
      auto issue_page = [&](int s, int i) {   // i = 0, 1, 2, ... in order
        if ((i >> 5) != cur_k) {
          curp = nxtp;
          ++cur_k;
          nxtp = page_of(cur_k + 1);
        }
        const int pp = __shfl_sync(0xffffffffu, curp, i & 31);
        fence_proxy_async();
        __syncwarp();
        if (lane == 0) {
          mbar_expect_tx(full_of(s), RB);
          bulk_load_hint(stage(s), rec_at<8>(sg, pp), RB, full_of(s), once);
        }
        pend |= 1u << s;
      };
      if (leader) {
        curp = page_of(0);
        nxtp = page_of(1);
        for (int i = 0; i < np && i < NS; ++i) {
          if (!claim(i)) { ok = false; break; }
          issue_page(i, i);
        }
      }
      for (int i = 0, s = 0; ok && i < np; ++i) {
        if (!wait_full(s)) { ok = false; break; }
        const char* rec = reinterpret_cast<const char*>(stage(s));
        const int tok0 = kP * (pg0 + i);
        if (tok0 + kP > free_end) fp8_page_mq<true>(rec, o, m, l, qa, zscale, tok0, lim_lo, lim_hi, T - tok0);
        else fp8_page_mq<false>(rec, o, m, l, qa, zscale, tok0, lim_lo, lim_hi, kP);
        release(s);
        if (leader && i + NS < np) {
          if (!claim(s)) { ok = false; break; }
          issue_page(s, i + NS);
        }
        s = s + 1 == NS ? 0 : s + 1;
      }
      if (!ok) {
        fail(b);
#pragma unroll
        for (int mt = 0; mt < 8; ++mt)
#pragma unroll
          for (int ct = 0; ct < 2; ++ct)
#pragma unroll
            for (int e = 0; e < 4; ++e) o[mt][ct][e] = 0.0f;
        m[0] = m[1] = -INFINITY;
        l[0] = l[1] = 0.0f;
      }
    }
    // every warp of the team is done reading the stages in its region before it
    // writes its scratch there (each warp passes these barriers once per segment)
    team_sync();
    // sums of columns gi, gi + 8 over the lane's four token positions
#pragma unroll
    for (int r = 0; r < 2; ++r) {
      l[r] += __shfl_xor_sync(0xffffffffu, l[r], 1);
      l[r] += __shfl_xor_sync(0xffffffffu, l[r], 2);
    }
    if (leader && seg_start >= r0 && lane == 0) {
      int ncon = 0;
      if (!own && slot_ok) ncon = owner_of(seg_end - 1, C, n_act) - gteam + 1;
      const long long first = 2LL * gteam + (seg_start <= r0 ? 0 : 1);
      meta_of(a)[static_cast<long long>(b) * a.H + h] =
          static_cast<long long>(static_cast<unsigned>(first)) | (static_cast<long long>(ncon) << 32);
    }
#pragma unroll
    for (int ct = 0; ct < 2; ++ct) {
      // column tile ct (columns 16 tile + 8 ct + j) in the two-columns-per-lane form of mma_to_gen
      MmaState ms;
#pragma unroll
      for (int mt = 0; mt < 8; ++mt)
#pragma unroll
        for (int e = 0; e < 4; ++e) ms.o[mt][e] = o[mt][ct][e] * vs;
#pragma unroll
      for (int k = 0; k < 4; ++k) ms.bias[k] = 0.0f;
      ms.m0 = __shfl_sync(0xffffffffu, m[ct], 8 * ti);
      ms.m1 = __shfl_sync(0xffffffffu, m[ct], 8 * ti + 4);
      const float lt0 = __shfl_sync(0xffffffffu, l[ct], 8 * ti), lt1 = __shfl_sync(0xffffffffu, l[ct], 8 * ti + 4);
      ms.l0 = lane < 4 ? lt0 : 0.0f;
      ms.l1 = lane < 4 ? lt1 : 0.0f;
      GenState gs;
      mma_to_gen(ms, gs, scratch);
      if (own || !slot_ok) {
#pragma unroll
        for (int j = 0; j < kNH; ++j) {
          const int c = 16 * tile + 8 * ct + j;
          if (c < cols) {
            const float inv = gs.l[j] > 0.0f ? 1.0f / gs.l[j] : 0.0f;
            store_out(a, row_of(c), lane,
                      make_float4(gs.o[j][0] * inv, gs.o[j][1] * inv, gs.o[j][2] * inv, gs.o[j][3] * inv));
          }
        }
      } else {
        const int k = seg_start <= r0 ? 0 : 1;
        float* P = a.ws + (2LL * gw + k) * partial_floats(a.pcols);
#pragma unroll
        for (int j = 0; j < kNH; ++j) {
          const int jj = 8 * ct + j;
          *reinterpret_cast<float4*>(P + jj * kD + 4 * lane) =
              make_float4(gs.o[j][0], gs.o[j][1], gs.o[j][2], gs.o[j][3]);
          if (lane == 0) {
            P[a.pcols * kD + 2 * jj] = gs.m[j];
            P[a.pcols * kD + 2 * jj + 1] = gs.l[j];
          }
        }
      }
    }
    fence_proxy_async();   // the scratch writes come before later bulk copies into the region
    team_sync();
    seg_start = seg_end;
    if (++h == a.H) {
      h = 0;
      if (++b >= a.B) break;
      sc = seg_cost<8>(a.seq_lens[b], a.R, a.tail_cost);
    }
  }
  if (pend) fail(-1);
}

// ---- multi-query over KIVI pages: each key group restored once to shared memory ----------
// A team restores each 32-token group once for all its columns: K^ = code * scale
// + min in fp32 (as the restore defines it), kept as an f16 high part plus the f16
// rest (about 22 bits; a key scale folded into the query in f16 would be the
// larger error on wide-scale channels), and V^ in f16. Keys past the quantized
// range come from the key ring (split the same way), values past it from the
// value ring, and tokens past T are zero. Each warp then runs plain MMAs from
// shared memory on its 16 (query, head) columns: the columns are the rows of the
// key-score MMA and the probabilities feed P V from registers, as for FP8 pages.
constexpr int kKRow = 2 * kD + 16;   // K^ rows, token-major: 272 B (ldmatrix rows in distinct banks)
constexpr int kVTRow = 2 * kG + 16;  // V^T rows, channel-major over a group's 32 tokens: 80 B
template <int BITS>
struct MqSmem {                      // byte offsets in a team's block of warp regions
  static constexpr int kStage = kStageBytesB<BITS>;   // two page records
  static constexpr int kKhi = 2 * kStage;
  static constexpr int kKlo = kKhi + kG * kKRow;
  static constexpr int kVt = kKlo + kG * kKRow;
  static constexpr int kEnd = kVt + kD * kVTRow;
};
constexpr int kMqMinTeam = (MqSmem<4>::kEnd + kRegion - 1) / kRegion;   // warps whose regions hold it
static_assert(MqSmem<4>::kStage % 16 == 0 && MqSmem<2>::kStage % 16 == 0 && MqSmem<4>::kEnd >= MqSmem<2>::kEnd,
              "16-byte aligned stages; 4-bit records take the most room");
static_assert(kMqMinTeam * 2 <= S4KV_DECODE_WARPS, "at least two restoring teams per CTA");

// byte of a key or value word that holds channel c_j (keys) / column j
__device__ __forceinline__ int byte_of_j(int j) { return j == 1 ? 2 : j == 2 ? 1 : j; }

// A code (0 .. 255) as a float, exactly: 2^23 + n holds n in its low mantissa bits.
__device__ __forceinline__ float code_f(uint32_t n) { return __fsub_rn(__uint_as_float(0x4B000000u | n), 8388608.0f); }

// High and low f16 parts of x: hi = x rounded to f16, lo = x - hi (exact in f32:
// the bits of x below hi's last place) rounded to f16, about 22 significant bits in
// all. x - hi is one mixed-precision FMA, hi (f16) times -1 plus x.
__device__ __forceinline__ void store_hi_lo(char* hi_row, char* lo_row, const float (&x)[8]) {
  const unsigned short neg1 = 0xBC00u;   // -1.0 in f16
  uint32_t h[4], r[4];
#pragma unroll
  for (int p = 0; p < 4; ++p) {
    h[p] = pack_f16x2(x[2 * p], x[2 * p + 1]);
    float l0, l1;
    asm("{\n\t.reg .b16 h0, h1;\n\tmov.b32 {h0, h1}, %2;\n\t"
        "fma.rn.f32.f16 %0, h0, %3, %4;\n\tfma.rn.f32.f16 %1, h1, %3, %5;\n\t}"
        : "=f"(l0), "=f"(l1)
        : "r"(h[p]), "h"(neg1), "f"(x[2 * p]), "f"(x[2 * p + 1]));
    r[p] = pack_f16x2(l0, l1);
  }
  *reinterpret_cast<uint4*>(hi_row) = make_uint4(h[0], h[1], h[2], h[3]);
  *reinterpret_cast<uint4*>(lo_row) = make_uint4(r[0], r[1], r[2], r[3]);
}

// Byte offsets of element (row r, column k) of the K-major f16 tcgen05 operands, in
// the swizzled layouts the tensor cores read at full shared-memory bandwidth (the
// tile starts on a 1024-byte boundary):
//  * K = 128 (channels), 128-byte swizzle: 64-element atoms along K, each a block of
//    `rows` rows of 128 bytes; the 16-byte chunk k / 8 of row r sits at chunk
//    (k / 8) xor (r mod 8) of the row;
//  * K = 32 (a group's tokens), 64-byte swizzle: rows of 64 bytes; chunk k / 8 sits
//    at chunk (k / 8) xor ((r / 2) mod 4).
__device__ __forceinline__ int sw128_off(int r, int k, int rows) {
  return (k >> 6) * rows * 128 + r * 128 + ((((k >> 3) & 7) ^ (r & 7)) << 4) + (k & 7) * 2;
}
__device__ __forceinline__ int sw64_off(int r, int k) {
  return r * 64 + ((((k >> 3) & 3) ^ ((r >> 1) & 3)) << 4) + (k & 7) * 2;
}

// Non-blocking test: has the phase of `parity` of the mbarrier completed?
__device__ __forceinline__ bool mbar_test(uint64_t* bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.test_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(smem_u32(bar)), "r"(parity)
      : "memory");
  return ok != 0;
}

// Bounded wait by non-blocking tests (never suspended by the barrier itself): true once
// the phase of `parity` has completed, false after `limit_ns` (0: give up at once).
// nap_ns > 0 sleeps that long between tests, leaving issue slots to other warps.
__device__ __forceinline__ bool mbar_poll(uint64_t* bar, uint32_t parity, long long limit_ns, unsigned nap_ns) {
  if (limit_ns <= 0) return false;
  if (mbar_test(bar, parity)) return true;
  const unsigned long long t0 = global_ns();
  for (unsigned it = 1;; ++it) {
    if (nap_ns) __nanosleep(nap_ns);
    if (mbar_test(bar, parity)) return true;
    if ((it & 15u) == 0 && static_cast<long long>(global_ns() - t0) > limit_ns) return false;
  }
}

// ---- tcgen05: 5th-generation tensor cores, accumulators in tensor memory -------------------
// Shared-memory operand descriptor of a swizzled K-major operand: start address / 16,
// leading byte offset 1 (unused by swizzled K-major layouts), stride byte offset / 16
// (the next 8 rows: 1024 for 128-byte rows, 512 for 64-byte rows), descriptor version
// 1, swizzle mode in bits 61-63 (2: 128-byte, 4: 64-byte). A K-step of 16 elements
// inside an atom advances the start address by 32 bytes.
constexpr uint32_t kSw128 = 2, kSw64 = 4;
__device__ __forceinline__ uint64_t umma_desc(uint32_t saddr, uint32_t sbo, uint32_t swizzle) {
  return static_cast<uint64_t>((saddr >> 4) & 0x3FFFu) | (static_cast<uint64_t>(1) << 16) |
         (static_cast<uint64_t>((sbo >> 4) & 0x3FFFu) << 32) | (static_cast<uint64_t>(1) << 46) |
         (static_cast<uint64_t>(swizzle) << 61);
}
// Instruction descriptor of kind::f16: f32 accumulator, f16 A and B, both K-major, N / 8, M / 16.
__host__ __device__ constexpr uint32_t umma_idesc(int M, int N) {
  return (1u << 4) | (static_cast<uint32_t>(N >> 3) << 17) | (static_cast<uint32_t>(M >> 4) << 24);
}
// D[tmem] (+)= A B^T, one thread issues; acc = false overwrites D.
__device__ __forceinline__ void umma_f16(uint32_t d_tmem, uint64_t a, uint64_t b, uint32_t idesc, bool acc) {
  asm volatile(
      "{\n\t.reg .pred p;\n\tsetp.ne.u32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
      "l"(a), "l"(b), "r"(idesc), "r"(acc ? 1u : 0u)
      : "memory");
}
// `bar` receives one arrival once the MMAs this thread issued so far have completed.
__device__ __forceinline__ void umma_commit(uint64_t* bar) {
  asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(smem_u32(bar))
               : "memory");
}
__device__ __forceinline__ void tc_fence_before() { asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void tc_fence_after() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }
// 32 consecutive 32-bit columns of this thread's TMEM lane (warp w addresses lanes 32 (w % 4) ..).
__device__ __forceinline__ void tmem_ld32(uint32_t taddr, uint32_t (&r)[32]) {
  asm volatile("tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
               : "r"(taddr));
}
__device__ __forceinline__ void tmem_st32(uint32_t taddr, const uint32_t (&r)[32]) {
  asm volatile("tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31,%32};" ::"r"(taddr), "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]), "r"(r[8]), "r"(r[9]), "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]), "r"(r[15]), "r"(r[16]), "r"(r[17]), "r"(r[18]), "r"(r[19]), "r"(r[20]), "r"(r[21]), "r"(r[22]), "r"(r[23]), "r"(r[24]), "r"(r[25]), "r"(r[26]), "r"(r[27]), "r"(r[28]), "r"(r[29]), "r"(r[30]), "r"(r[31]) : "memory");
}
__device__ __forceinline__ void tmem_wait_ld() { asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory"); }
__device__ __forceinline__ void tmem_wait_st() { asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory"); }

// Keys of group tokens t0 .. t0 + 31: thread thr of nthr takes (token, 8 channels)
// items. kTail: a token may be past the quantized keys (ring) or past T (zero).
// kCore: K^ in the 128-byte swizzled layout (rows = tokens, K = channels), else rows of kKRow.
// kStack (with kCore): high and low parts in one 64-row tile at khi, the high
// parts in rows 0..31 and the low parts in rows 32..63 (klo is not used).
// key_item: the 8 keys of item it (token tau, channels c0 ..).
template <int BITS, bool kTail, bool kCore>
__device__ __forceinline__ void key_item(const char* stage, int it, int t0, int T, int Tk, const uint16_t* kring,
                                         int dtype, int& tau, int& c0, float (&x)[8]) {
  using F = Rec<BITS>;
  constexpr int RS = kRecStrideB<BITS>;
  // core layout: consecutive threads take consecutive tokens (conflict-free stores)
  tau = kCore ? (it & 31) : (it >> 4);
  c0 = 8 * (kCore ? (it >> 5) : (it & 15));
  const int t = t0 + tau;
  if (!kTail || t < Tk) {
    // channel 32 b + 4 kk + j: slices kk0 (j = 0..3 of c0..c0+3) and kk0 + 1 (c0+4..c0+7)
    const char* rec = stage + (tau >> 4) * RS;
    const int tp = tau & 15, hi = tp >> 3, L = 4 * (tp & 7) + (c0 >> 5), kk0 = (c0 & 31) >> 2;
    uint32_t code[8];
    if constexpr (BITS == 4) {
      const uint2 w = *reinterpret_cast<const uint2*>(rec + F::kKc + (kk0 >> 2) * 512 + L * 16 + (kk0 & 3) * 4);
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        code[j] = (w.x >> (8 * byte_of_j(j) + 4 * hi)) & 15;
        code[4 + j] = (w.y >> (8 * byte_of_j(j) + 4 * hi)) & 15;
      }
    } else {
      const uint32_t w = *reinterpret_cast<const uint32_t*>(rec + F::kKc + L * 16 + (kk0 >> 1) * 4);
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        code[j] = (w >> (8 * byte_of_j(j) + 2 * hi)) & 3;
        code[4 + j] = (w >> (8 * byte_of_j(j) + 2 * (2 + hi))) & 3;
      }
    }
    // scale / min of channels c0 .. c0 + 7 in the group's page of channel half c0 / 64
    const char* mrec = stage + (c0 >> 6) * RS + F::kKm;
    const int cl = c0 & 63, u = cl >> 5, i0 = (cl & 31) >> 2;
    const float4 sa = *reinterpret_cast<const float4*>(mrec + (2 * i0 + u) * 16);
    const float4 sb = *reinterpret_cast<const float4*>(mrec + (2 * i0 + 2 + u) * 16);
    const float4 ma = *reinterpret_cast<const float4*>(mrec + 256 + (2 * i0 + u) * 16);
    const float4 mb = *reinterpret_cast<const float4*>(mrec + 256 + (2 * i0 + 2 + u) * 16);
    const float sc[8] = {sa.x, sa.y, sa.z, sa.w, sb.x, sb.y, sb.z, sb.w};
    const float mn[8] = {ma.x, ma.y, ma.z, ma.w, mb.x, mb.y, mb.z, mb.w};
#pragma unroll
    for (int j = 0; j < 8; ++j) x[j] = fmaf(code_f(code[j]), sc[j], mn[j]);
  } else if (t < T) {
    const uint4 r = *reinterpret_cast<const uint4*>(kring + static_cast<long long>(t % kG) * kD + c0);
    const uint32_t rw[4] = {r.x, r.y, r.z, r.w};
#pragma unroll
    for (int p = 0; p < 4; ++p) {
      x[2 * p] = widen16(static_cast<uint16_t>(rw[p] & 0xffff), dtype);
      x[2 * p + 1] = widen16(static_cast<uint16_t>(rw[p] >> 16), dtype);
    }
  } else {
#pragma unroll
    for (int j = 0; j < 8; ++j) x[j] = 0.0f;
  }
}

template <bool kCore, bool kStack>
__device__ __forceinline__ void key_store(char* khi, char* klo, int tau, int c0, const float (&x)[8]) {
  const int off = kCore ? sw128_off(tau, c0, kStack ? 2 * kG : kG) : tau * kKRow + 2 * c0;
  if constexpr (kStack) store_hi_lo(khi + off, khi + sw128_off(kG + tau, c0, 2 * kG), x);
  else store_hi_lo(khi + off, klo + off, x);
}

template <int BITS, bool kTail>
__device__ void restore_key_pairs(const char* stage, char* kt, int t0, int T, int Tk, const uint16_t* kring,
                                  int dtype, int thr, int nthr) {
  constexpr int kItems = kG * 16;
  // Core layout: an item is a code word's two tokens (page token tp and tp + 8 of record
  // r) x 8 channels, so its metadata loads and index arithmetic serve 16 keys. Lanes
  // take 8 tokens of 4 channel octets: the 16-byte stores of a quarter warp go to 8
  // rows whose swizzled chunks differ. A group's keys are all quantized (t0 < Tk) or
  // all ring rows: Tk and t0 are multiples of 32.
  using F = Rec<BITS>;
  constexpr int RS = kRecStrideB<BITS>;
  const bool quant = !kTail || t0 < Tk;
  for (int kp = thr; kp < kItems / 2; kp += nthr) {
    const int r = kp >> 7, c0 = 8 * ((kp >> 3) & 15), tp = kp & 7;
    const char* rec = stage + r * RS;
    const int L = 4 * tp + (c0 >> 5), kk0 = (c0 & 31) >> 2;
    uint32_t code[2][8];   // [token tp, tp + 8][channel c0 + j]
    float sc[8], mn[8];
    if (quant) {
      if constexpr (BITS == 4) {
        const uint2 w = *reinterpret_cast<const uint2*>(rec + F::kKc + (kk0 >> 2) * 512 + L * 16 + (kk0 & 3) * 4);
#pragma unroll
        for (int hh = 0; hh < 2; ++hh)
#pragma unroll
          for (int j = 0; j < 4; ++j) {
            code[hh][j] = (w.x >> (8 * byte_of_j(j) + 4 * hh)) & 15;
            code[hh][4 + j] = (w.y >> (8 * byte_of_j(j) + 4 * hh)) & 15;
          }
      } else {
        const uint32_t w = *reinterpret_cast<const uint32_t*>(rec + F::kKc + L * 16 + (kk0 >> 1) * 4);
#pragma unroll
        for (int hh = 0; hh < 2; ++hh)
#pragma unroll
          for (int j = 0; j < 4; ++j) {
            code[hh][j] = (w >> (8 * byte_of_j(j) + 2 * hh)) & 3;
            code[hh][4 + j] = (w >> (8 * byte_of_j(j) + 2 * (2 + hh))) & 3;
          }
      }
      // scale / min of channels c0 .. c0 + 7 in the group's page of channel half c0 / 64
      const char* mrec = stage + (c0 >> 6) * RS + F::kKm;
      const int cl = c0 & 63, u = cl >> 5, i0 = (cl & 31) >> 2;
      const float4 sa = *reinterpret_cast<const float4*>(mrec + (2 * i0 + u) * 16);
      const float4 sb = *reinterpret_cast<const float4*>(mrec + (2 * i0 + 2 + u) * 16);
      const float4 ma = *reinterpret_cast<const float4*>(mrec + 256 + (2 * i0 + u) * 16);
      const float4 mb = *reinterpret_cast<const float4*>(mrec + 256 + (2 * i0 + 2 + u) * 16);
      sc[0] = sa.x; sc[1] = sa.y; sc[2] = sa.z; sc[3] = sa.w; sc[4] = sb.x; sc[5] = sb.y; sc[6] = sb.z; sc[7] = sb.w;
      mn[0] = ma.x; mn[1] = ma.y; mn[2] = ma.z; mn[3] = ma.w; mn[4] = mb.x; mn[5] = mb.y; mn[6] = mb.z; mn[7] = mb.w;
    }
    uint4 ring[2];   // the two tokens' ring rows (channels c0 ..), loaded together
    if (!quant) {
#pragma unroll
      for (int hh = 0; hh < 2; ++hh) {
        const int t = t0 + 16 * r + tp + 8 * hh;
        ring[hh] = t < T ? *reinterpret_cast<const uint4*>(kring + static_cast<long long>(t % kG) * kD + c0)
                         : make_uint4(0u, 0u, 0u, 0u);
      }
    }
#pragma unroll
    for (int hh = 0; hh < 2; ++hh) {
      const int tau = 16 * r + tp + 8 * hh, t = t0 + tau;
      float x[8];
      if (quant) {
#pragma unroll
        for (int j = 0; j < 8; ++j) x[j] = fmaf(code_f(code[hh][j]), sc[j], mn[j]);
      } else if (t < T) {
        const uint4 rw4 = ring[hh];
        const uint32_t rw[4] = {rw4.x, rw4.y, rw4.z, rw4.w};
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          x[2 * q] = widen16(static_cast<uint16_t>(rw[q] & 0xffff), dtype);
          x[2 * q + 1] = widen16(static_cast<uint16_t>(rw[q] >> 16), dtype);
        }
      } else {
#pragma unroll
        for (int j = 0; j < 8; ++j) x[j] = 0.0f;
      }
      key_store<true, true>(kt, kt, tau, c0, x);
    }
  }
}

template <int BITS, bool kTail, bool kCore = false, bool kStack = false>
__device__ void restore_keys(const char* stage, char* khi, char* klo, int t0, int T, int Tk,
                             const uint16_t* kring, int dtype, int thr, int nthr) {
  constexpr int kItems = kG * 16;
  static_assert(!kCore || kStack, "the core layout stacks the high and low parts");
  if constexpr (!kCore) {   // the register-bound kernel: one item at a time
    for (int it = thr; it < kItems; it += nthr) {
      int tau, c0;
      float x[8];
      key_item<BITS, kTail, kCore>(stage, it, t0, T, Tk, kring, dtype, tau, c0, x);
      key_store<kCore, kStack>(khi, klo, tau, c0, x);
    }
  } else {
    restore_key_pairs<BITS, kTail>(stage, khi, t0, T, Tk, kring, dtype, thr, nthr);
  }
}

// Values of the group into V^T (channel-major): thread thr of nthr takes code
// words (a word holds 4 tokens of 2 channels at 4 bits, of 4 channels at 2 bits).
// kTail: a token may be past the quantized values (ring) or past T (zero).
// kCore: V^ (rows = channels, K = the group's tokens) in the 64-byte swizzled layout.
// value_item: the values of word item it, v[channel slot][byte].
template <int BITS>
constexpr int kValueWords = (BITS == 4 ? 8 : 4) * 32;   // code words per page
template <int BITS, bool kTail>
__device__ __forceinline__ void value_item(const char* stage, int it, int t0, int T, int Tv, const uint16_t* vring,
                                           int R, int dtype, float (&v)[BITS == 4 ? 2 : 4][4]) {
  using F = Rec<BITS>;
  constexpr int RS = kRecStrideB<BITS>;
  constexpr int kWords = kValueWords<BITS>;
  constexpr int kCh = BITS == 4 ? 2 : 4;             // channels per byte
  const int p = it / kWords, wi = it % kWords;
  const int L = wi & 31, mw = wi >> 5;              // word (mt or mp, L)
  const int a = L >> 2, b = L & 3;
  const int tb = t0 + 16 * p;                       // first token of the page
  const char* rec = stage + p * RS;
  // byte i of the word holds page token tok[i]; e[i]: its entry in the metadata quad
  const int tok[4] = {2 * b, 2 * b + 8, 2 * b + 1, 2 * b + 9};
  const int e[4] = {0, 2, 1, 3};
  const bool quant = !kTail || tb < Tv;             // any token of the page quantized
  uint32_t w = 0;
  float4 s4 = make_float4(0.0f, 0.0f, 0.0f, 0.0f), m4 = s4;
  if (quant) {
    const int k = BITS == 4 ? (mw >> 1) : mw;       // value group of the word's channels
    w = BITS == 4 ? *reinterpret_cast<const uint32_t*>(rec + F::kVc + (mw >> 2) * 512 + L * 16 + (mw & 3) * 4)
                  : *reinterpret_cast<const uint32_t*>(rec + F::kVc + L * 16 + mw * 4);
    s4 = *reinterpret_cast<const float4*>(rec + F::kVm + ((2 * k) * 4 + b) * 16);
    m4 = *reinterpret_cast<const float4*>(rec + F::kVm + ((2 * k + 1) * 4 + b) * 16);
  }
  const float sq[4] = {s4.x, s4.y, s4.z, s4.w}, mq[4] = {m4.x, m4.y, m4.z, m4.w};
  uint16_t rv[4][kCh];   // residual rows of the word's ring tokens, loaded before their first use
  if constexpr (kTail) {
#pragma unroll
    for (int i = 0; i < 4; ++i)
#pragma unroll
      for (int q = 0; q < kCh; ++q) {
        const int t = tb + tok[i];
        const int ch = BITS == 4 ? 16 * mw + a + 8 * q : 32 * mw + 8 * q + a;
        rv[i][q] = t >= Tv && t < T ? vring[static_cast<long long>(t % R) * kD + ch] : static_cast<uint16_t>(0);
      }
  }
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const int t = tb + tok[i];
#pragma unroll
    for (int q = 0; q < kCh; ++q) {
      float x = 0.0f;
      if (!kTail || t < Tv) {
        const uint32_t code = BITS == 4 ? (w >> (8 * i + 4 * q)) & 15u : (w >> (8 * i + 2 * q)) & 3u;
        x = fmaf(code_f(code), sq[e[i]], mq[e[i]]);
      } else if (t < T) {
        x = widen16(rv[i][q], dtype);
      }
      v[q][i] = x;
    }
  }
}

template <int BITS, bool kCore>
__device__ __forceinline__ void value_store(char* vt, int it, const float (&v)[BITS == 4 ? 2 : 4][4]) {
  constexpr int kWords = kValueWords<BITS>;
  constexpr int kCh = BITS == 4 ? 2 : 4;
  const int p = it / kWords, wi = it % kWords;
  const int L = wi & 31, mw = wi >> 5;
  const int a = L >> 2, b = L & 3;
#pragma unroll
  for (int q = 0; q < kCh; ++q) {
    const int ch = BITS == 4 ? 16 * mw + a + 8 * q : 32 * mw + 8 * q + a;
    const int tk = 16 * p + 2 * b;
    // tokens 2b, 2b + 1 and 2b + 8, 2b + 9 of page p
    char* r0 = vt + (kCore ? sw64_off(ch, tk) : ch * kVTRow + 2 * tk);
    char* r1 = vt + (kCore ? sw64_off(ch, tk + 8) : ch * kVTRow + 2 * (tk + 8));
    *reinterpret_cast<uint32_t*>(r0) = pack_f16x2(v[q][0], v[q][2]);
    *reinterpret_cast<uint32_t*>(r1) = pack_f16x2(v[q][1], v[q][3]);
  }
}

// 4 bits, core layout: an item is two adjacent code words (mw even and mw + 1, one
// 8-byte load) of the same 32-channel value group, so they share the 4 tokens' scale
// and min loads.
template <bool kTail>
__device__ void restore_value_pairs(const char* stage, char* vt, int t0, int T, int Tv, const uint16_t* vring,
                                    int R, int dtype, int thr, int nthr) {
  using F = Rec<4>;
  constexpr int RS = kRecStrideB<4>;
  constexpr int kWords = kValueWords<4>;
  for (int vq = thr; vq < kWords; vq += nthr) {
    const int p = vq >> 7, k = (vq >> 5) & 3, L = vq & 31;   // page, value group (words 2k, 2k + 1), lane word
    const int a = L >> 2, b = L & 3;
    const int tb = t0 + 16 * p;
    const char* rec = stage + p * RS;
    const int tok[4] = {2 * b, 2 * b + 8, 2 * b + 1, 2 * b + 9};
    const int e[4] = {0, 2, 1, 3};
    const bool quant = !kTail || tb < Tv;
    uint2 w = make_uint2(0u, 0u);
    float4 s4 = make_float4(0.0f, 0.0f, 0.0f, 0.0f), m4 = s4;
    if (quant) {
      w = *reinterpret_cast<const uint2*>(rec + F::kVc + (k >> 1) * 512 + L * 16 + (k & 1) * 8);
      s4 = *reinterpret_cast<const float4*>(rec + F::kVm + ((2 * k) * 4 + b) * 16);
      m4 = *reinterpret_cast<const float4*>(rec + F::kVm + ((2 * k + 1) * 4 + b) * 16);
    }
    const float sq[4] = {s4.x, s4.y, s4.z, s4.w}, mq[4] = {m4.x, m4.y, m4.z, m4.w};
    // residual rows of the item's ring tokens, all loads issued before their first use
    uint16_t rv[2][4][2];
    if constexpr (kTail) {
#pragma unroll
      for (int h = 0; h < 2; ++h)
#pragma unroll
        for (int i = 0; i < 4; ++i)
#pragma unroll
          for (int q = 0; q < 2; ++q) {
            const int t = tb + tok[i];
            rv[h][i][q] = t >= Tv && t < T ? vring[static_cast<long long>(t % R) * kD + 16 * (2 * k + h) + a + 8 * q]
                                           : static_cast<uint16_t>(0);
          }
    }
#pragma unroll
    for (int h = 0; h < 2; ++h) {   // word mw = 2 k + h
      const int mw = 2 * k + h;
      const uint32_t wd = h ? w.y : w.x;
      float v[2][4];
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const int t = tb + tok[i];
#pragma unroll
        for (int q = 0; q < 2; ++q) {
          float x = 0.0f;
          if (!kTail || t < Tv) {
            x = fmaf(code_f((wd >> (8 * i + 4 * q)) & 15u), sq[e[i]], mq[e[i]]);
          } else if (t < T) {
            x = widen16(rv[h][i][q], dtype);
          }
          v[q][i] = x;
        }
      }
      value_store<4, true>(vt, p * kWords + 32 * mw + L, v);
    }
  }
}
template <int BITS, bool kTail, bool kCore = false>
__device__ void restore_values(const char* stage, char* vt, int t0, int T, int Tv, const uint16_t* vring, int R,
                               int dtype, int thr, int nthr) {
  constexpr int kItems = 2 * kValueWords<BITS>;
  if constexpr (!kCore || BITS == 2) {
    // one word item at a time: the register-bound kernel, or 2 bits (a word holds a
    // whole value group's 4 channels)
    for (int it = thr; it < kItems; it += nthr) {
      float v[BITS == 4 ? 2 : 4][4];
      value_item<BITS, kTail>(stage, it, t0, T, Tv, vring, R, dtype, v);
      value_store<BITS, kCore>(vt, it, v);
    }
  } else {
    restore_value_pairs<kTail>(stage, vt, t0, T, Tv, vring, R, dtype, thr, nthr);
  }
}

// An FP8 group (tokens t0 .. t0 + 31: two page records in the stage) into the
// swizzled tiles of the tcgen05 kernel: K^ (rows = tokens, K = channels) and
// V^ (rows = channels, K = tokens). E4M3 codes widen to f16 exactly; the per-head
// scales stay outside (the key scale joins the softmax scale, the value scale
// the output). Tokens at or past nvalid = T - t0 are zero: a partial last page
// holds stale bytes, and a group's absent second page was not copied.
__device__ void convert_fp8_group(const char* stage, char* kt, char* vt, int nvalid, int thr, int nthr) {
  constexpr int RS = kRecStrideB<8>;
  constexpr int kKeyWords = 2 * 128, kValueQuads = 2 * 32;   // per group: 16-byte key words, 64-byte value quads
  for (int it = thr; it < kKeyWords + kValueQuads; it += nthr) {
    if (it < kKeyWords) {
      // key word (page p, kp, L = 4 a + b): channels 32 b + 8 kp .. + 7 of page tokens
      // a and a + 8; its 32-bit word e holds channels 2e, 2e + 1 of token a in the
      // low half and of token a + 8 in the high half
      const int p = it >> 7, kp = (it >> 5) & 3, L = it & 31, a = L >> 2, bq = L & 3;
      const int tau = 16 * p + a, c0 = 32 * bq + 8 * kp;
      uint4 w = make_uint4(0u, 0u, 0u, 0u);
      if (tau < nvalid) w = *reinterpret_cast<const uint4*>(stage + p * RS + kp * 512 + L * 16);
      const uint32_t e[4] = {w.x, w.y, w.z, w.w};
      uint32_t lo[4], hi[4];
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        lo[k] = fp8x2_to_f16x2(e[k] & 0xffffu);
        hi[k] = tau + 8 < nvalid ? fp8x2_to_f16x2(e[k] >> 16) : 0u;
      }
      *reinterpret_cast<uint4*>(kt + sw128_off(tau, c0, kG)) = make_uint4(lo[0], lo[1], lo[2], lo[3]);
      *reinterpret_cast<uint4*>(kt + sw128_off(tau + 8, c0, kG)) = make_uint4(hi[0], hi[1], hi[2], hi[3]);
    } else {
      // value quad (page p, kp, a): words L = 4 a + b, b = 0 .. 3, hold channels
      // 32 kp + 16 u + 8 up + a (u, up = 0, 1) of the page's 16 tokens; in word b,
      // 32-bit word 2 u + w, half up, holds tokens 2 b + 8 w and 2 b + 8 w + 1
      const int v = it - kKeyWords, p = v >> 5, kp = (v >> 3) & 3, a = v & 7;
      const int tb = 16 * p;
      uint4 wd[4];
#pragma unroll
      for (int b = 0; b < 4; ++b)
        wd[b] = tb < nvalid ? *reinterpret_cast<const uint4*>(stage + p * RS + 2048 + kp * 512 + 64 * a + 16 * b)
                            : make_uint4(0u, 0u, 0u, 0u);
#pragma unroll
      for (int u = 0; u < 2; ++u) {
#pragma unroll
        for (int w = 0; w < 2; ++w) {
#pragma unroll
          for (int up = 0; up < 2; ++up) {
            uint32_t chunk[4];
#pragma unroll
            for (int b = 0; b < 4; ++b) {
              const uint32_t words[4] = {wd[b].x, wd[b].y, wd[b].z, wd[b].w};
              uint32_t x = fp8x2_to_f16x2((words[2 * u + w] >> (16 * up)) & 0xffffu);
              const int t = tb + 8 * w + 2 * b;   // the pair's first token in the group
              if (t >= nvalid) x = 0u;
              else if (t + 1 >= nvalid) x &= 0xffffu;
              chunk[b] = x;
            }
            const int ch = 32 * kp + 16 * u + 8 * up + a;
            *reinterpret_cast<uint4*>(vt + sw64_off(ch, tb + 8 * w)) =
                make_uint4(chunk[0], chunk[1], chunk[2], chunk[3]);
          }
        }
      }
    }
  }
}

// One restored group for a warp's 16 columns (rows gi: column c_lo, gi + 8:
// c_hi): scores from K^ (high and low parts) by MMA, causal mask (kMask: the
// group reaches some column's limit), lazy online softmax, P V from V^T.
template <bool kMask>
__device__ __forceinline__ void mq_group_mma(uint32_t khi, uint32_t klo, uint32_t vt, float (&o)[8][2][4],
                                             float (&m)[2], float (&l)[2], const uint32_t (&qa)[8][4],
                                             float scale, int t0, int lim_lo, int lim_hi) {
  const int lane = threadIdx.x & 31, ti = lane & 3;
  const int j = lane >> 3, r = lane & 7;
  // ldmatrix rows: K^ token 8 (j / 2) + r, channels + 8 (j % 2); V^T channel 8 (j % 2) + r, tokens + 8 (j / 2)
  const uint32_t kofs = (8 * (j >> 1) + r) * kKRow + 16 * (j & 1);
  const uint32_t vofs = (8 * (j & 1) + r) * kVTRow + 16 * (j >> 1);
  float acc[4][4];
#pragma unroll
  for (int nt = 0; nt < 4; ++nt)
#pragma unroll
    for (int e = 0; e < 4; ++e) acc[nt][e] = 0.0f;
#pragma unroll
  for (int kk = 0; kk < 8; ++kk) {
    uint32_t h0[4], h1[4], l0[4], l1[4];   // tokens 0-15 and 16-31: {b0, b1} of two n8 tiles each
    ldsm_x4(khi + kofs + 32 * kk, h0);
    ldsm_x4(khi + kofs + 16 * kKRow + 32 * kk, h1);
    ldsm_x4(klo + kofs + 32 * kk, l0);
    ldsm_x4(klo + kofs + 16 * kKRow + 32 * kk, l1);
    mma16816(acc[0], qa[kk], h0[0], h0[1]);
    mma16816(acc[1], qa[kk], h0[2], h0[3]);
    mma16816(acc[2], qa[kk], h1[0], h1[1]);
    mma16816(acc[3], qa[kk], h1[2], h1[3]);
    mma16816(acc[0], qa[kk], l0[0], l0[1]);
    mma16816(acc[1], qa[kk], l0[2], l0[3]);
    mma16816(acc[2], qa[kk], l1[0], l1[1]);
    mma16816(acc[3], qa[kk], l1[2], l1[3]);
  }
  // z[row][tile][x]: column row (0: c_lo, 1: c_hi), token t0 + 8 tile + 2 ti + x
  float z[2][4][2];
#pragma unroll
  for (int nt = 0; nt < 4; ++nt) {
    z[0][nt][0] = acc[nt][0] * scale;
    z[0][nt][1] = acc[nt][1] * scale;
    z[1][nt][0] = acc[nt][2] * scale;
    z[1][nt][1] = acc[nt][3] * scale;
    if (kMask) {
#pragma unroll
      for (int x = 0; x < 2; ++x) {
        const int t = t0 + 8 * nt + 2 * ti + x;
        z[0][nt][x] = t < lim_lo ? z[0][nt][x] : -INFINITY;
        z[1][nt][x] = t < lim_hi ? z[1][nt][x] : -INFINITY;
      }
    }
  }
  float mx[2];
#pragma unroll
  for (int rw = 0; rw < 2; ++rw) {
    mx[rw] = z[rw][0][0];
#pragma unroll
    for (int nt = 0; nt < 4; ++nt) mx[rw] = fmaxf(mx[rw], fmaxf(z[rw][nt][0], z[rw][nt][1]));
    mx[rw] = fmaxf(mx[rw], __shfl_xor_sync(0xffffffffu, mx[rw], 1));
    mx[rw] = fmaxf(mx[rw], __shfl_xor_sync(0xffffffffu, mx[rw], 2));
  }
  if (__any_sync(0xffffffffu, mx[0] > m[0] + kLazy || mx[1] > m[1] + kLazy)) {
    float al[2];
#pragma unroll
    for (int rw = 0; rw < 2; ++rw) {
      const float mn = fmaxf(m[rw], mx[rw]);
      al[rw] = mn == -INFINITY ? 1.0f : ex2(m[rw] - mn);
      m[rw] = mn;
      l[rw] *= al[rw];
    }
#pragma unroll
    for (int ct = 0; ct < 2; ++ct) {
      const float a0 = __shfl_sync(0xffffffffu, al[ct], 8 * ti);
      const float a1 = __shfl_sync(0xffffffffu, al[ct], 8 * ti + 4);
#pragma unroll
      for (int mt = 0; mt < 8; ++mt) {
        o[mt][ct][0] *= a0;
        o[mt][ct][1] *= a1;
        o[mt][ct][2] *= a0;
        o[mt][ct][3] *= a1;
      }
    }
  }
  uint32_t pb[2][4][1];   // packed p: [row][tile] (tokens 2ti, 2ti + 1 of the tile)
#pragma unroll
  for (int rw = 0; rw < 2; ++rw) {
    float sum = 0.0f;
#pragma unroll
    for (int nt = 0; nt < 4; ++nt) {
      const float p0 = z[rw][nt][0] == -INFINITY ? 0.0f : ex2(z[rw][nt][0] - m[rw]);
      const float p1 = z[rw][nt][1] == -INFINITY ? 0.0f : ex2(z[rw][nt][1] - m[rw]);
      sum += p0 + p1;
      pb[rw][nt][0] = pack_f16x2(p0, p1);
    }
    l[rw] += sum;
  }
#pragma unroll
  for (int pg = 0; pg < 2; ++pg) {
#pragma unroll
    for (int mt = 0; mt < 8; ++mt) {
      uint32_t av[4];   // V^T of channels 16 mt .. + 15, tokens 16 pg .. + 15
      ldsm_x4(vt + vofs + 16 * mt * kVTRow + 32 * pg, av);
      mma16816(o[mt][0], av, pb[0][2 * pg][0], pb[0][2 * pg + 1][0]);
      mma16816(o[mt][1], av, pb[1][2 * pg][0], pb[1][2 * pg + 1][0]);
    }
  }
}

// Multi-query attention over KIVI pages (4- or 2-bit), the same causal reading
// and cost line as mq_kernel: teams of tw = max(kMqMinTeam, ceil(nq g / 16)) warps.
// Per key group: the leader's bounded wait on the group's records (its outcome
// shared through shared memory), the team restores the group, the leader stages
// the group two ahead, the column warps run mq_group_mma. Named team barriers
// separate the phases; every warp of a team passes each barrier equally often.
template <int BITS>
__global__ void __launch_bounds__(32 * S4KV_DECODE_WARPS, S4KV_DECODE_MIN_CTAS) mqd_kernel(DecodeArgs a) {
  using F = Rec<BITS>;
  using M = MqSmem<BITS>;
  constexpr int kWarps = S4KV_DECODE_WARPS;
  constexpr int kThreads = 32 * kWarps;
  using SmemT = Smem<kWarps>;
  extern __shared__ __align__(128) uint8_t smem_raw[];
  SmemT& sm = *reinterpret_cast<SmemT*>(smem_raw);
  long long* pre = reinterpret_cast<long long*>(smem_raw + prefix_offset<0>());   // [B + 1]
  __shared__ int team_ok[kWarps];
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int tw = a.tw, tpc = kWarps / tw;
  const int team = warp / tw, tile = warp - team * tw;
  const bool in_team = team < tpc;
  const int lead = in_team ? team * tw : warp;
  const bool leader = in_team && tile == 0;
  const int cols = a.nq * a.g;
  const int ncw = (cols + 15) / 16;   // warps with columns; the others only restore
  const bool colw = tile < ncw;
  char* blk = reinterpret_cast<char*>(sm.region[lead]);   // the team's regions, contiguous
  float* scratch = reinterpret_cast<float*>(sm.region[warp]);
  uint64_t* full = sm.bar[lead];

  if (leader && lane == 0) {
    mbar_init(&full[0], 1);
    mbar_init(&full[1], 1);
  }
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  {
    long long carry = 0;
    __shared__ long long wt[kWarps];
    for (int base = 0; base < a.B; base += kThreads) {
      const int b = base + tid;
      const long long cnt = b < a.B ? a.H * seg_cost(a.seq_lens[b], a.R, a.tail_cost).cost : 0;
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
  int n_act = static_cast<int>(gridDim.x) * tpc;
  if (a.max_warps > 0 && a.max_warps < n_act) n_act = a.max_warps;   // the option caps teams here
  {
    const long long cap = (C + kMinUnits - 1) / kMinUnits;
    if (cap < n_act) n_act = static_cast<int>(cap);
  }
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  if (!in_team) return;
  const int gteam = blockIdx.x * tpc + team;
  if (gteam >= n_act) return;
  const int gw = blockIdx.x * kWarps + warp;
  const long long r0 = gteam * C / n_act, r1 = (gteam + 1) * C / n_act;
  const uint64_t once = policy_evict_first();
  const int gi = lane >> 2, ti = lane & 3;
  const int thr = 32 * tile + lane, nthr = 32 * tw;
  auto team_sync = [&]() {   // named barrier of the team (id 0 is __syncthreads); tw >= 3
    asm volatile("bar.sync %0, %1;" ::"r"(1 + team), "r"(32 * tw) : "memory");
  };
  uint32_t fph = 0, pend = 0;   // leader: stage parities and copies in flight
  bool aborted = false;

  int b;
  {
    int lo = 0, hi = a.B - 1;
    while (lo < hi) {
      const int mid = (lo + hi + 1) >> 1;
      if (pre[mid] <= r0) lo = mid; else hi = mid - 1;
    }
    b = lo;
  }
  SegCost sc = seg_cost(a.seq_lens[b], a.R, a.tail_cost);
  int h = static_cast<int>((r0 - pre[b]) / sc.cost);
  long long seg_start = pre[b] + h * sc.cost;

  while (seg_start < r1) {
    const long long seg_end = seg_start + sc.cost;
    const int T = max(a.seq_lens[b], 0);
    const long long lo = max(r0, seg_start) - seg_start, hi = min(r1, seg_end) - seg_start;
    const bool own = lo == 0 && hi == sc.cost;
    const int nm = sc.main_groups;
    const int u0 = static_cast<int>(lo < nm ? lo : nm), u1 = static_cast<int>(hi < nm ? hi : nm);
    int c0 = 0, c1 = 0;
    if (sc.tail_chunks > 0 && hi > nm) {
      c0 = static_cast<int>(lo > nm ? (lo - nm + a.tail_cost - 1) / a.tail_cost : 0);
      const long long cc = (hi - nm + a.tail_cost - 1) / a.tail_cost;
      c1 = static_cast<int>(cc < sc.tail_chunks ? cc : sc.tail_chunks);
    }
    const int nmain = u1 - u0, ng = nmain + (c1 - c0);
    auto group_of = [&](int i) { return i < nmain ? u0 + i : nm + c0 + (i - nmain); };
    const int slot = a.slot_ids ? a.slot_ids[b] : b;
    const bool slot_ok = slot >= 0 && slot < a.max_slots;
    const bool table_ok = static_cast<long long>(a.bt_stride) * kP >= T;
    const int lens_v = slot_ok ? a.lens[slot * a.H + h] : 0;
    Seg sg;
    sg.pages = a.pages;
    sg.bt = a.block_table + static_cast<long long>(b) * a.bt_stride;
    sg.H = a.H;
    sg.h = h;
    sg.T = T;
    const int npT = (T + kP - 1) / kP;
    const int Tk = T & ~(kG - 1), Tv = max(0, T - a.R);
    const uint16_t* kring = reinterpret_cast<const uint16_t*>(a.kring) + (slot_ok ? slot : 0) * a.kring_slot + h * a.kring_head;
    const uint16_t* vring = reinterpret_cast<const uint16_t*>(a.vring) + (slot_ok ? slot : 0) * a.vring_slot + h * a.vring_head;
    bool valid = slot_ok && T > 0;
    bool bad = false;
    if (valid && table_ok && ng > 0) {
      const int p_lo = 2 * group_of(0), p_hi = min(2 * group_of(ng - 1) + 2, npT);
      for (int base = p_lo; base < p_hi; base += 32 * 8) {
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
    } else if (lens_v != T || T > a.max_seq_len || T < a.nq) {
      valid = false;
      if (lane == 0) report(a.status, S4KV_ERR_DEVICE, S4KV_DEV_BAD_LENGTH, b);
    } else if (!table_ok) {
      valid = false;
      if (lane == 0) report(a.status, S4KV_ERR_DEVICE, S4KV_DEV_BAD_TABLE, b);
    }
    valid = valid && !__any_sync(0xffffffffu, bad) && !aborted;
    auto row_of = [&](int c) -> long long {
      return (static_cast<long long>(b) * a.nq + c / a.g) * a.Hq + h * a.g + c % a.g;
    };
    float o[8][2][4];
#pragma unroll
    for (int mt = 0; mt < 8; ++mt)
#pragma unroll
      for (int ct = 0; ct < 2; ++ct)
#pragma unroll
        for (int e = 0; e < 4; ++e) o[mt][ct][e] = 0.0f;
    float m[2] = {-INFINITY, -INFINITY}, l[2] = {0.0f, 0.0f};
    if (valid && ng > 0) {
      const int c_lo = 16 * tile + gi, c_hi = c_lo + 8;
      uint32_t qa[8][4];   // A operand: columns c_lo (rows gi), c_hi (rows gi + 8); channels 16 kk + 2 ti (+1, +8, +9)
#pragma unroll
      for (int kk = 0; kk < 8; ++kk)
#pragma unroll
        for (int e = 0; e < 4; ++e) qa[kk][e] = 0u;
      if (colw) {
        const uint32_t* qlo = c_lo < cols ? reinterpret_cast<const uint32_t*>(a.q + row_of(c_lo) * kD) : nullptr;
        const uint32_t* qhi = c_hi < cols ? reinterpret_cast<const uint32_t*>(a.q + row_of(c_hi) * kD) : nullptr;
        auto f16w = [&](uint32_t w) -> uint32_t {   // two query values as f16x2 (bf16 widened, then rounded: exact)
          if (a.dtype == S4KV_F16) return w;
          return pack_f16x2(widen16(static_cast<uint16_t>(w & 0xffff), S4KV_BF16),
                            widen16(static_cast<uint16_t>(w >> 16), S4KV_BF16));
        };
#pragma unroll
        for (int kk = 0; kk < 8; ++kk) {
          const int wc = 8 * kk + ti;   // word of channels 16 kk + 2 ti, + 1
          if (qlo) {
            qa[kk][0] = f16w(qlo[wc]);
            qa[kk][2] = f16w(qlo[wc + 4]);
          }
          if (qhi) {
            qa[kk][1] = f16w(qhi[wc]);
            qa[kk][3] = f16w(qhi[wc + 4]);
          }
        }
      }
      const int lim_lo = c_lo < cols ? T - a.nq + c_lo / a.g + 1 : T;
      const int lim_hi = c_hi < cols ? T - a.nq + c_hi / a.g + 1 : T;
      int free_end = min(lim_lo, lim_hi);   // groups ending at or before it need no mask
#pragma unroll
      for (int x = 1; x < 32; x <<= 1) free_end = min(free_end, __shfl_xor_sync(0xffffffffu, free_end, x));
      const uint32_t khi_s = smem_u32(blk + M::kKhi), klo_s = smem_u32(blk + M::kKlo), vt_s = smem_u32(blk + M::kVt);
      auto issue = [&](int s, int i) {   // leader: the records of group i into stage s
        const int g = group_of(i);
        const int np = 32 * g + kP < T ? 2 : 1;
        const int p0 = sg.bt[2 * g], p1 = np == 2 ? sg.bt[2 * g + 1] : p0;
        fence_proxy_async();
        __syncwarp();
        if (lane == 0) {
          char* dst = blk + s * M::kStage;
          mbar_expect_tx(&full[s], np * F::kBytes);
          bulk_load_hint(dst, rec_at<BITS>(sg, p0), F::kBytes, &full[s], once);
          if (np == 2) bulk_load_hint(dst + kRecStrideB<BITS>, rec_at<BITS>(sg, p1), F::kBytes, &full[s], once);
        }
        pend |= 1u << s;
      };
      if (leader) {
        for (int i = 0; i < ng && i < 2; ++i) issue(i, i);
      }
      for (int i = 0; i < ng; ++i) {
        const int s = i & 1;
        if (leader) {
          const bool got = __all_sync(0xffffffffu, mbar_wait(&full[s], (fph >> s) & 1u, a.wait_ns));
          if (got) {
            fph ^= 1u << s;
            pend &= ~(1u << s);
          }
          if (lane == 0) team_ok[team] = got ? 1 : 0;
        }
        team_sync();
        if (!team_ok[team]) {   // the same outcome for every warp of the team
          aborted = true;
          break;
        }
        if (!leader) {   // the phase has completed: this wait orders the records' bytes for this warp
          mbar_wait(&full[s], (fph >> s) & 1u, kDrainNs);
          fph ^= 1u << s;
        }
        const int g = group_of(i), t0 = 32 * g;
        const char* stage = blk + s * M::kStage;
        if (t0 + kG <= min(Tk, Tv)) {
          restore_keys<BITS, false>(stage, blk + M::kKhi, blk + M::kKlo, t0, T, Tk, kring, a.dtype, thr, nthr);
          restore_values<BITS, false>(stage, blk + M::kVt, t0, T, Tv, vring, a.R, a.dtype, thr, nthr);
        } else {
          restore_keys<BITS, true>(stage, blk + M::kKhi, blk + M::kKlo, t0, T, Tk, kring, a.dtype, thr, nthr);
          restore_values<BITS, true>(stage, blk + M::kVt, t0, T, Tv, vring, a.R, a.dtype, thr, nthr);
        }
        fence_proxy_async();   // the stage's generic reads come before its next bulk copy
        team_sync();
        if (leader && i + 2 < ng) issue(s, i + 2);
        if (colw) {
          const float scale = a.sm_scale_log2;
          if (t0 + kG > free_end) mq_group_mma<true>(khi_s, klo_s, vt_s, o, m, l, qa, scale, t0, lim_lo, lim_hi);
          else mq_group_mma<false>(khi_s, klo_s, vt_s, o, m, l, qa, scale, t0, lim_lo, lim_hi);
        }
        team_sync();   // the restored group is free again
      }
      if (aborted) {
        if (leader) {
          if (lane == 0) report(a.status, S4KV_ERR_DEVICE_TIMEOUT, S4KV_DEV_TIMEOUT, b);
          for (int s = 0; s < 2; ++s) {
            if ((pend >> s) & 1u) {
              mbar_wait(&full[s], (fph >> s) & 1u, kDrainNs);
              fph ^= 1u << s;
              pend &= ~(1u << s);
            }
          }
        }
#pragma unroll
        for (int mt = 0; mt < 8; ++mt)
#pragma unroll
          for (int ct = 0; ct < 2; ++ct)
#pragma unroll
            for (int e = 0; e < 4; ++e) o[mt][ct][e] = 0.0f;
        m[0] = m[1] = -INFINITY;
        l[0] = l[1] = 0.0f;
      }
    }
    // every warp passes these two barriers once per segment: the team is done with
    // the stages and the restored group before warps write scratch in their regions
    team_sync();
#pragma unroll
    for (int rw = 0; rw < 2; ++rw) {
      l[rw] += __shfl_xor_sync(0xffffffffu, l[rw], 1);
      l[rw] += __shfl_xor_sync(0xffffffffu, l[rw], 2);
    }
    if (leader && seg_start >= r0 && lane == 0) {
      int ncon = 0;
      if (!own && slot_ok) ncon = owner_of(seg_end - 1, C, n_act) - gteam + 1;
      const long long first = 2LL * gteam + (seg_start <= r0 ? 0 : 1);
      meta_of(a)[static_cast<long long>(b) * a.H + h] =
          static_cast<long long>(static_cast<unsigned>(first)) | (static_cast<long long>(ncon) << 32);
    }
    if (colw) {
#pragma unroll
      for (int ct = 0; ct < 2; ++ct) {
        MmaState ms;
#pragma unroll
        for (int mt = 0; mt < 8; ++mt)
#pragma unroll
          for (int e = 0; e < 4; ++e) ms.o[mt][e] = o[mt][ct][e];
#pragma unroll
        for (int k = 0; k < 4; ++k) ms.bias[k] = 0.0f;
        ms.m0 = __shfl_sync(0xffffffffu, m[ct], 8 * ti);
        ms.m1 = __shfl_sync(0xffffffffu, m[ct], 8 * ti + 4);
        const float lt0 = __shfl_sync(0xffffffffu, l[ct], 8 * ti), lt1 = __shfl_sync(0xffffffffu, l[ct], 8 * ti + 4);
        ms.l0 = lane < 4 ? lt0 : 0.0f;
        ms.l1 = lane < 4 ? lt1 : 0.0f;
        GenState gs;
        mma_to_gen(ms, gs, scratch);
        if (own || !slot_ok) {
#pragma unroll
          for (int jj = 0; jj < kNH; ++jj) {
            const int c = 16 * tile + 8 * ct + jj;
            if (c < cols) {
              const float inv = gs.l[jj] > 0.0f ? 1.0f / gs.l[jj] : 0.0f;
              store_out(a, row_of(c), lane,
                        make_float4(gs.o[jj][0] * inv, gs.o[jj][1] * inv, gs.o[jj][2] * inv, gs.o[jj][3] * inv));
            }
          }
        } else {
          const int k = seg_start <= r0 ? 0 : 1;
          float* P = a.ws + (2LL * gw + k) * partial_floats(a.pcols);
#pragma unroll
          for (int jj = 0; jj < kNH; ++jj) {
            const int cc = 8 * ct + jj;
            *reinterpret_cast<float4*>(P + cc * kD + 4 * lane) =
                make_float4(gs.o[jj][0], gs.o[jj][1], gs.o[jj][2], gs.o[jj][3]);
            if (lane == 0) {
              P[a.pcols * kD + 2 * cc] = gs.m[jj];
              P[a.pcols * kD + 2 * cc + 1] = gs.l[jj];
            }
          }
        }
      }
    }
    fence_proxy_async();   // the scratch writes come before later bulk copies into the region
    team_sync();
    seg_start = seg_end;
    if (++h == a.H) {
      h = 0;
      if (++b >= a.B) break;
      sc = seg_cost(a.seq_lens[b], a.R, a.tail_cost);
    }
  }
  if (pend) {   // never expected: every issued copy is waited for
    for (int s = 0; s < 2; ++s)
      if ((pend >> s) & 1u) mbar_wait(&full[s], (fph >> s) & 1u, kDrainNs);
  }
}

// Multi-query attention on tcgen05, warp-specialized. The CTA is one team and
// works through its slice of the cost line segment by segment:
//  * warps 4 .. 9 restore each key group into one of four slots of swizzled
//    tiles (K^ high and low parts stacked as 64 rows, V^); warp 10 stages page
//    records four (FP8: six) groups ahead, with the pool pages of the next 32
//    groups held in registers;
//  * warp 11 issues the MMAs: S[slot] = Q K^T (M = 128 query columns, N = 64:
//    the group's 32 tokens' high parts, then their low parts; FP8: N = 32, K =
//    128) into the slot's tensor-memory buffer once the slot is restored, and
//    O += P V (N = 128 channels, K = 32 tokens) once P is written, whichever of
//    the two is possible first;
//  * warps 0 .. 3 read S one query column per thread (TMEM lane), add the two
//    halves, run the lazy online softmax, rescale their O rows in tensor memory
//    when the maximum moves, and write P into one of two buffers.
// Hand-offs are mbarriers (tcgen05.commit for the MMAs) waited on with a bound; a
// wait that runs out raises a shared flag and every role leaves its loop. The only
// CTA-wide barriers sit between the roles' loops, reached by every thread once per
// segment; the mbarriers are re-initialised between segments, when nothing is in
// flight. Tensor memory is allocated after the CTA-uniform exit and freed on the
// only way out.
// FP8 pages (BITS = 8) take the same pipeline: the producing warps widen each
// group's codes to f16 tiles (exact, so no low part and no second key MMA), the
// key scale joins the softmax scale and the value scale multiplies the output.
// Softmax warps whose 32 columns are all past the call's columns only keep P zero.
// Tuning of the tcgen05 multi-query kernel (mqt_kernel) and of the multi-query merge.
#ifndef S4KV_MQT_PBUFS
#define S4KV_MQT_PBUFS 2   // P buffers
#endif
#ifndef S4KV_MQT_WARPS
#define S4KV_MQT_WARPS 12   // warps of a CTA on KIVI pages
#endif
#ifndef S4KV_MQT_WARPS_FP8
#define S4KV_MQT_WARPS_FP8 14   // warps of a CTA on FP8 pages
#endif
#ifndef S4KV_MQT_TAIL_WEIGHT
#define S4KV_MQT_TAIL_WEIGHT 5   // tail-chunk weight on KIVI pages: this / 3 times the decode weight
#endif
#ifndef S4KV_MQT_SLOTS
#define S4KV_MQT_SLOTS 4   // restored groups in flight on KIVI pages
#endif
#ifndef S4KV_MQT_REC_STAGES
#define S4KV_MQT_REC_STAGES 4   // record stages on KIVI pages
#endif
#ifndef S4KV_MQT_NAP_NS
#define S4KV_MQT_NAP_NS 64   // restoring warps' sleep between tests of a barrier
#endif
#ifndef S4KV_MQT_POLL_NS
#define S4KV_MQT_POLL_NS 32   // loading and MMA warps' sleep between polling rounds
#endif
#ifndef S4KV_MQ_MERGE_BLOCKS
#define S4KV_MQ_MERGE_BLOCKS 16   // merge blocks per attention CTA of a multi-query call
#endif
// Tracing builds: per-group event times of each warp of the tcgen05 kernel, after the
// trace words in the workspace (a warp slot's words: restore, score and P V issue
// times of its first groups).
constexpr int kMqTimelineWords = kTraceWords ? 128 : 0;

__host__ __device__ constexpr int mqt_warps(int bits) { return bits == 8 ? S4KV_MQT_WARPS_FP8 : S4KV_MQT_WARPS; }

template <int BITS>
__global__ void __launch_bounds__(32 * mqt_warps(BITS), 1) mqt_kernel(DecodeArgs a) {
  constexpr int kWarps = mqt_warps(BITS);
  constexpr int kThreads = 32 * kWarps;
  static_assert(kWarps >= 12 && kWarps <= 16, "4 softmax warps, 6 to 10 restoring warps, a loading warp and an MMA warp");
  constexpr int kProd0 = 4, kProdWarps = kWarps - 6, kLoadWarp = kWarps - 2, kMmaWarp = kWarps - 1;
  // partial results and trace words are laid out per S4KV_DECODE_WARPS warps of a CTA
  constexpr int kSlotWarps = S4KV_DECODE_WARPS;
  static_assert(kSlotWarps >= 8, "a CTA's 8 partial slots (two per softmax warp)");
  using F = Rec<BITS>;
  using SmemT = Smem<kSlotWarps>;
  constexpr int kStage = kStageBytesB<BITS>;
  constexpr int kRecStages = BITS == 8 ? 6 : S4KV_MQT_REC_STAGES, kSlots = BITS == 8 ? 4 : S4KV_MQT_SLOTS;   // records staged ahead; restored groups in flight
  constexpr int kQ = (kRecStages * kStage + 1023) / 1024 * 1024;   // Q: 128 columns x 128 channels
  constexpr int kTile = kG * kD * 2;                       // one 32 x 128 f16 tile
  constexpr int kTps = BITS == 8 ? 2 : 3;                  // tiles a slot: K^ (hi), [K^ lo,] V^
  constexpr int kSlot0 = kQ + 128 * kD * 2;                // slot s at kSlot0 + kTps s kTile
  constexpr int kPo = kSlot0 + kTps * kSlots * kTile;      // P[b]: 128 columns x 32 tokens, kPBufs buffers
  constexpr int kPTile = 128 * kG * 2;
  constexpr int kPBufs = S4KV_MQT_PBUFS;
  static_assert(kPBufs >= 2, "the softmax of group i overlaps the P V MMA of group i - 1");
  // the tiles take the whole decode layout (warp regions, P tiles and barrier words,
  // none used here as such), from a 1024-byte boundary
  static_assert(kPo + kPBufs * kPTile + 1024 <= static_cast<int>(sizeof(SmemT)), "tiles fit the shared window");
  // S[s] of a KIVI group holds the scores of the keys' high parts (32 columns) and of
  // their low parts (32 more): one N = 64 MMA per K-step over the stacked key tile
  constexpr int kSCols = BITS == 8 ? kG : 2 * kG;
  constexpr uint32_t kTmemCols = BITS == 8 ? 256 : 512;    // O in columns 0 .. 127, S[s] at 128 + kSCols s
  static_assert(128 + kSCols * kSlots <= static_cast<int>(kTmemCols), "S buffers fit the allocation");
  enum { kRecFull = 0, kSlotReady = kRecStages, kSFull = kSlotReady + kSlots, kSlotFree = kSFull + kSlots,
         kPReady = kSlotFree + kSlots, kPvDone = kPReady + kPBufs, kNumBars = kPvDone + kPBufs };
  static_assert(kNumBars <= 32, "one phase bit per mbarrier");
  extern __shared__ __align__(128) uint8_t smem_raw[];
  SmemT& sm = *reinterpret_cast<SmemT*>(smem_raw);
  S4KV_TRACE(const unsigned long long t_entry = global_ns();)
  long long* pre = reinterpret_cast<long long*>(smem_raw + prefix_offset<0>());   // [B + 1]
  __shared__ uint32_t tmem_slot;
  __shared__ __align__(8) uint64_t bars[kNumBars];
  __shared__ int abort_flag;
  // swizzled tiles start on 1024-byte boundaries of the shared window
  char* base = reinterpret_cast<char*>(sm.region[0]) + ((1024u - (smem_u32(sm.region[0]) & 1023u)) & 1023u);
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  // Softmax warps whose 32 columns all lie past the call's columns (at most 64
  // columns leave warps 2 and 3 without work) restore groups instead: nlive softmax
  // warps, nprod restoring warps (warps 4 .. 9 and the spare softmax warps).
  const int nlive = min(4, (a.nq * a.g + 31) / 32);
  const int nprod = kProdWarps + (4 - nlive);
  const bool producer = (warp >= kProd0 && warp < kProd0 + kProdWarps) || (warp < 4 && warp >= nlive);
  const int prank = warp >= kProd0 ? warp - kProd0 : kProdWarps + (warp - nlive);   // producers only
  auto init_bars = [&]() {   // thread 0
    for (int k = 0; k < kRecStages; ++k) mbar_init(&bars[kRecFull + k], 1);
    for (int k = 0; k < kSlots; ++k) {
      mbar_init(&bars[kSlotReady + k], nprod);
      mbar_init(&bars[kSFull + k], 1);
      mbar_init(&bars[kSlotFree + k], 1);
    }
    for (int k = 0; k < kPBufs; ++k) {
      mbar_init(&bars[kPReady + k], nlive);
      mbar_init(&bars[kPvDone + k], 1);
    }
  };
  {
    long long carry = 0;
    __shared__ long long wt[kWarps];
    for (int base_b = 0; base_b < a.B; base_b += kThreads) {
      const int b = base_b + tid;
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
  int n_act = static_cast<int>(gridDim.x);   // one team per CTA
  if (a.max_warps > 0 && a.max_warps < n_act) n_act = a.max_warps;
  {
    const long long cap = (C + kMinUnits - 1) / kMinUnits;
    if (cap < n_act) n_act = static_cast<int>(cap);
  }
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  const int gteam = blockIdx.x;
  if (gteam >= n_act) return;   // CTA-uniform, before tensor memory is allocated

  if (tid == 0) {
    init_bars();
    abort_flag = 0;
  }
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  if (warp == 0) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(&tmem_slot)),
                 "n"(kTmemCols));
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;");
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = tmem_slot;
  const uint32_t t_row = static_cast<uint32_t>(32 * (warp & 3)) << 16;   // softmax warp's TMEM lanes
  volatile int* flag = &abort_flag;

  const long long r0 = gteam * C / n_act, r1 = (gteam + 1) * C / n_act;
  const uint64_t once = policy_evict_first();
  const int cols = a.nq * a.g;
  const float scale = a.sm_scale_log2;
  const uint32_t q_s = smem_u32(base + kQ), p_s = smem_u32(base + kPo);
  uint32_t ph = 0;     // this thread's phase bit of each mbarrier
  int n_copies = 0;   // loading warp: groups whose records were sent for (0 .. n_copies - 1)
  bool aborted = false;
  // warp-uniform bounded wait; false (and the flag raised) when it runs out or the
  // flag is already up
  // tracing builds: per warp [0] span, [1] first wait, [2] second wait, [3] work, [4] groups,
  // [5] .. [7] absolute entry, loop start and end
  // (tracing builds: the loading and MMA warps take the last two trace slots of the
  // CTA, restoring warps past the slots before them share the last of those)
  S4KV_TRACE(const int tslot = warp >= kLoadWarp ? kSlotWarps - (kWarps - warp) : min(warp, kSlotWarps - 3);)
  S4KV_TRACE(unsigned long long tq[5] = {global_ns(), 0, 0, 0, 0}; unsigned long long tmark = 0;
             unsigned long long* tl_out = reinterpret_cast<unsigned long long*>(meta_of(a) + meta_words(a.B, a.H)) +
                                          static_cast<long long>(gridDim.x) * kSlotWarps * (kTraceWords + 4) +
                                          (static_cast<long long>(blockIdx.x) * kSlotWarps + tslot) * kMqTimelineWords;
             int tl_n = 0, tl_m = 0;
             auto tl = [&](int k) { if (lane == 0 && k < kMqTimelineWords) tl_out[k] = global_ns(); };)
  // Waits test the barrier without suspending on it: the softmax warps (the critical
  // path) spin, the other roles nap between tests so that they leave issue slots to
  // the softmax warps sharing their sub-partitions.
  const unsigned nap = warp < nlive ? 0u : static_cast<unsigned>(S4KV_MQT_NAP_NS);
  auto wait_w = [&](int k) -> bool {
    if (__shfl_sync(0xffffffffu, *flag, 0)) return false;
    const uint32_t par = (ph >> k) & 1u;
    const bool ok = __all_sync(0xffffffffu, mbar_poll(&bars[k], par, a.wait_ns, nap));
    if (ok) ph ^= 1u << k;
    else if (lane == 0) *flag = 1;
    return ok;
  };

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
    const long long seg_end = seg_start + sc.cost;
    const int T = max(a.seq_lens[b], 0);
    const long long lo = max(r0, seg_start) - seg_start, hi = min(r1, seg_end) - seg_start;
    const bool own = lo == 0 && hi == sc.cost;
    const int nm = sc.main_groups;
    const int u0 = static_cast<int>(lo < nm ? lo : nm), u1 = static_cast<int>(hi < nm ? hi : nm);
    int c0 = 0, c1 = 0;
    if (sc.tail_chunks > 0 && hi > nm) {
      c0 = static_cast<int>(lo > nm ? (lo - nm + a.tail_cost - 1) / a.tail_cost : 0);
      const long long cc = (hi - nm + a.tail_cost - 1) / a.tail_cost;
      c1 = static_cast<int>(cc < sc.tail_chunks ? cc : sc.tail_chunks);
    }
    const int nmain = u1 - u0, ng = nmain + (c1 - c0);
    auto group_of = [&](int i) { return i < nmain ? u0 + i : nm + c0 + (i - nmain); };
    const int slot = a.slot_ids ? a.slot_ids[b] : b;
    const bool slot_ok = slot >= 0 && slot < a.max_slots;
    const bool table_ok = static_cast<long long>(a.bt_stride) * kP >= T;
    const int lens_v = slot_ok ? a.lens[slot * a.H + h] : 0;
    Seg sg;
    sg.pages = a.pages;
    sg.bt = a.block_table + static_cast<long long>(b) * a.bt_stride;
    sg.H = a.H;
    sg.h = h;
    sg.T = T;
    const int npT = (T + kP - 1) / kP;
    const int Tk = T & ~(kG - 1), Tv = max(0, T - a.R);
    const uint16_t* kring = reinterpret_cast<const uint16_t*>(a.kring) + (slot_ok ? slot : 0) * a.kring_slot + h * a.kring_head;
    const uint16_t* vring = reinterpret_cast<const uint16_t*>(a.vring) + (slot_ok ? slot : 0) * a.vring_slot + h * a.vring_head;
    bool valid = slot_ok && T > 0;
    bool bad = false;
    if (warp == 0 && valid && table_ok && ng > 0) {
      const int p_lo = 2 * group_of(0), p_hi = min(2 * group_of(ng - 1) + 2, npT);
      for (int pb = p_lo; pb < p_hi; pb += 32 * 8) {
        int pp[8];
#pragma unroll
        for (int k = 0; k < 8; ++k) {
          const int lp = pb + 32 * k + lane;
          pp[k] = lp < p_hi ? sg.bt[lp] : 0;
        }
#pragma unroll
        for (int k = 0; k < 8; ++k) {
          if (pb + 32 * k + lane < p_hi && (pp[k] < 0 || pp[k] >= a.num_pages)) {
            bad = true;
            report(a.status, S4KV_ERR_DEVICE, S4KV_DEV_BAD_PAGE, pp[k]);
          }
        }
      }
    }
    if (!slot_ok) {
      if (tid == 0) report(a.status, S4KV_ERR_DEVICE, S4KV_DEV_BAD_SLOT, slot);
    } else if (lens_v != T || T > a.max_seq_len || T < a.nq) {
      valid = false;
      if (tid == 0) report(a.status, S4KV_ERR_DEVICE, S4KV_DEV_BAD_LENGTH, b);
    } else if (!table_ok) {
      valid = false;
      if (tid == 0) report(a.status, S4KV_ERR_DEVICE, S4KV_DEV_BAD_TABLE, b);
    }
    valid = !__syncthreads_or(bad) && valid && !aborted;   // the same for every thread
    auto row_of = [&](int c) -> long long {
      return (static_cast<long long>(b) * a.nq + c / a.g) * a.Hq + h * a.g + c % a.g;
    };
    const int r = tid;   // softmax warps: query column of this thread
    const int lim = r < cols ? T - a.nq + r / a.g + 1 : T;
    // FP8 pages: the head's key scale joins the softmax scale, its value scale the output
    const float zs = BITS == 8 ? scale * a.fp8_scale[h] : scale;
    const float vsc = BITS == 8 ? a.fp8_scale[a.H + h] : 1.0f;
    const int free_end = T - a.nq + 1;   // groups ending by then need no causal mask
    float m_r = -INFINITY, l_r = 0.0f;
    ph = 0;   // the mbarriers start this segment freshly initialised
    if (valid && ng > 0) {
      for (int it = tid; it < 128 * 16; it += kThreads) {   // Q: zero past cols
        const int row = it & 127, c0q = 8 * (it >> 7);
        uint4 v = make_uint4(0u, 0u, 0u, 0u);
        if (row < cols) {
          v = *reinterpret_cast<const uint4*>(a.q + row_of(row) * kD + c0q);
          if (a.dtype == S4KV_BF16) {
            uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
            for (int k = 0; k < 4; ++k)
              w[k] = pack_f16x2(widen16(static_cast<uint16_t>(w[k] & 0xffff), S4KV_BF16),
                                widen16(static_cast<uint16_t>(w[k] >> 16), S4KV_BF16));
            v = make_uint4(w[0], w[1], w[2], w[3]);
          }
        }
        *reinterpret_cast<uint4*>(base + kQ + sw128_off(row, c0q, 128)) = v;
      }
      fence_proxy_async();
      __syncthreads();
      // loading warp: pool pages of groups 32 k + lane (both records), a batch of 32 groups
      // held in registers ahead of the copies that need them
      auto pages_of = [&](int k, int& x0, int& x1) {
        const int i = 32 * k + lane;
        x0 = x1 = 0;
        if (i < ng) {
          const int g = group_of(i);
          x0 = sg.bt[2 * g];
          x1 = 32 * g + kP < T ? sg.bt[2 * g + 1] : x0;
        }
      };
      int cur0 = 0, cur1 = 0, nxt0 = 0, nxt1 = 0, cur_k = 0;
      auto issue = [&](int i) {   // loading warp: the records of group i into record stage i % kRecStages
        if ((i >> 5) != cur_k) {
          cur0 = nxt0;
          cur1 = nxt1;
          ++cur_k;
          pages_of(cur_k + 1, nxt0, nxt1);
        }
        const int p0 = __shfl_sync(0xffffffffu, cur0, i & 31), p1 = __shfl_sync(0xffffffffu, cur1, i & 31);
        const int s = i % kRecStages;
        const int np = 32 * group_of(i) + kP < T ? 2 : 1;
        fence_proxy_async();
        __syncwarp();
        if (lane == 0) {
          char* dst = base + s * kStage;
          mbar_expect_tx(&bars[kRecFull + s], np * F::kBytes);
          bulk_load_hint(dst, rec_at<BITS>(sg, p0), F::kBytes, &bars[kRecFull + s], once);
          if (np == 2) bulk_load_hint(dst + kRecStrideB<BITS>, rec_at<BITS>(sg, p1), F::kBytes, &bars[kRecFull + s], once);
        }
        n_copies = i + 1;
      };
      auto qk = [&](int i) {   // S[i % kSlots] = Q K^T of group i
        const int s = i % kSlots;
        tc_fence_after();
        if (lane == 0) {
          const uint32_t kh_s = smem_u32(base + kSlot0 + kTps * s * kTile);
          const uint32_t d = tmem + 128 + kSCols * s;
          // K-step j: atom j / 4 (Q: 128 rows; K^: kSCols rows of 128 bytes, the 32 high
          // parts then, on KIVI pages, the 32 low parts), 32 bytes per step inside it.
          // FP8 keys are exact in f16: no low part.
#pragma unroll
          for (int j = 0; j < 8; ++j)
            umma_f16(d, umma_desc(q_s + (j >> 2) * 128 * 128 + (j & 3) * 32, 1024, kSw128),
                     umma_desc(kh_s + (j >> 2) * kSCols * 128 + (j & 3) * 32, 1024, kSw128),
                     umma_idesc(128, kSCols), j > 0);
          umma_commit(&bars[kSFull + s]);
        }
        __syncwarp();
      };
      auto pv = [&](int i) {   // O += P V of group i (slot i % kSlots, P buffer i % kPBufs)
        tc_fence_after();
        if (lane == 0) {
          const uint32_t v_s = smem_u32(base + kSlot0 + kTps * (i % kSlots) * kTile + (kTps - 1) * kTile);
          const uint32_t pb = p_s + (i % kPBufs) * kPTile;
#pragma unroll
          for (int j = 0; j < 2; ++j)
            umma_f16(tmem, umma_desc(pb + 32 * j, 512, kSw64), umma_desc(v_s + 32 * j, 512, kSw64),
                     umma_idesc(128, kD), i > 0 || j > 0);
          umma_commit(&bars[kSlotFree + i % kSlots]);
          umma_commit(&bars[kPvDone + i % kPBufs]);
        }
        __syncwarp();
      };
      auto ready = [&](int k) -> bool {   // lane 0 tests mbarrier k's phase; warp-uniform
        const bool got = __shfl_sync(0xffffffffu, lane == 0 ? mbar_test(&bars[k], (ph >> k) & 1u) : false, 0);
        if (got) ph ^= 1u << k;
        return got;
      };
      if (warp == kLoadWarp) {
        // ---- loading warp ----
        // The records of group i + kRecStages go into the stage of group i once
        // every restoring warp is done with it (its arrival on the slot's barrier).
        // This warp also issues the P V MMAs: issuing a tcgen05.mma holds the issuing
        // thread for about the instruction's run, so the score MMAs go from the MMA
        // warp and these from here, and neither waits behind the other.
        // Each barrier is observed once a phase, in group order, and never two phases
        // late: P of group i + kPBufs waits for P V of group i (issued here after seeing P
        // of group i), and slot i is restored again only after P V of group i, which is
        // issued here only after seeing slot i's first restore (i < ncopy) unless no
        // more copies are to come.
        pages_of(0, cur0, cur1);
        pages_of(1, nxt0, nxt1);
        for (int i = 0; i < ng && i < kRecStages; ++i) issue(i);
        int ncopy = 0, npv = 0;   // stages refilled past the first kRecStages; P V issued
        unsigned long long t_last = global_ns();
        for (unsigned spins = 0; npv < ng || ncopy + kRecStages < ng;) {
          bool did = false;
          if (ncopy + kRecStages < ng && ready(kSlotReady + ncopy % kSlots)) {
            issue(ncopy + kRecStages);
            ++ncopy;
            did = true;
          }
          if (npv < ng && (npv < ncopy || ncopy + kRecStages >= ng) && ready(kPReady + npv % kPBufs)) {
            S4KV_TRACE(if (tl_n < 64) tl(tl_n);)
            pv(npv++);
            S4KV_TRACE(if (tl_n < 64) tl(64 + tl_n++);)
            did = true;
          }
          if (did) {
            t_last = global_ns();
            spins = 0;
            continue;
          }
          if ((++spins & 15u) == 0) {
            if (__shfl_sync(0xffffffffu, *flag, 0)) break;
            if (static_cast<long long>(global_ns() - t_last) > a.wait_ns) {
              if (lane == 0) *flag = 1;
              break;
            }
          }
          __nanosleep(S4KV_MQT_POLL_NS);
        }
      } else if (producer) {
        // ---- restoring warps ----
        const int pt = 32 * prank + lane, npt = 32 * nprod;
        if (warp < 4) {
          // a spare softmax warp: its rows of every P buffer stay zero for the segment
          // (its columns are past the call's; the P V MMAs read every row)
#pragma unroll
          for (int bf = 0; bf < kPBufs; ++bf)
#pragma unroll
            for (int kg = 0; kg < 4; ++kg)
              *reinterpret_cast<uint4*>(base + kPo + bf * kPTile + sw64_off(tid, 8 * kg)) = make_uint4(0u, 0u, 0u, 0u);
          fence_proxy_async();   // before the P V MMAs read them (ordered by this warp's slot arrivals)
        }
        for (int i = 0; i < ng; ++i) {
          const int s = i % kSlots, rs = i % kRecStages;
          S4KV_TRACE(tmark = global_ns();)
          if (i >= kSlots && !wait_w(kSlotFree + s)) break;   // P V of group i - kSlots done with slot s
          S4KV_TRACE({ const unsigned long long x = global_ns(); tq[1] += x - tmark; tmark = x; tl(3 * tl_n); })
          if (!wait_w(kRecFull + rs)) break;
          S4KV_TRACE({ const unsigned long long x = global_ns(); tq[2] += x - tmark; tmark = x; tl(3 * tl_n + 1); })
          const int g = group_of(i), t0 = 32 * g;
          const char* stage = base + rs * kStage;
          char* tiles = base + kSlot0 + kTps * s * kTile;
          if constexpr (BITS == 8) {
            convert_fp8_group(stage, tiles, tiles + kTile, T - t0, pt, npt);
          } else if (t0 + kG <= min(Tk, Tv)) {
            restore_keys<BITS, false, true, true>(stage, tiles, tiles, t0, T, Tk, kring, a.dtype, pt, npt);
            restore_values<BITS, false, true>(stage, tiles + 2 * kTile, t0, T, Tv, vring, a.R, a.dtype, pt, npt);
          } else {
            restore_keys<BITS, true, true, true>(stage, tiles, tiles, t0, T, Tk, kring, a.dtype, pt, npt);
            restore_values<BITS, true, true>(stage, tiles + 2 * kTile, t0, T, Tv, vring, a.R, a.dtype, pt, npt);
          }
          fence_proxy_async();   // tile writes before the MMAs; stage reads before its next copy
          __syncwarp();
          if (lane == 0) asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(&bars[kSlotReady + s])) : "memory");
          S4KV_TRACE(tq[3] += global_ns() - tmark; tq[4] += 1; tl(3 * tl_n + 2); ++tl_n;)
        }
      } else if (warp == kMmaWarp) {
        // ---- MMA warp: the score MMAs ----
        // S = Q K^T of group j needs slot j restored, and S buffer j % kSlots read by
        // the softmax of group j - kSlots. The slot's barrier carries both: restoring
        // group j waited for P V of group j - kSlots to complete, which was issued only
        // once the softmax of that group had read its S and written P. Bounded like
        // every wait: no progress for the wait limit, or the flag raised by another
        // role, ends the loop.
        int nqk = 0;
        unsigned long long t_last = global_ns();
        S4KV_TRACE(unsigned long long t_idle0 = 0;)
        for (unsigned spins = 0; nqk < ng;) {
          bool did = false;
          if (ready(kSlotReady + nqk % kSlots)) {
            S4KV_TRACE(if (tl_n < 64) tl(tl_n);)
            qk(nqk++);
            S4KV_TRACE(if (tl_n < 64) tl(64 + tl_n++);)
            did = true;
          }
          if (did) {
            S4KV_TRACE(if (t_idle0) { tq[1] += global_ns() - t_idle0; t_idle0 = 0; } tq[4] += 1;)
            t_last = global_ns();
            spins = 0;
            continue;
          }
          S4KV_TRACE(if (!t_idle0) t_idle0 = global_ns();)
          if ((++spins & 15u) == 0) {
            if (__shfl_sync(0xffffffffu, *flag, 0)) break;
            if (static_cast<long long>(global_ns() - t_last) > a.wait_ns) {
              if (lane == 0) *flag = 1;
              break;
            }
          }
          __nanosleep(S4KV_MQT_POLL_NS);
        }
      } else if (warp < 4) {
        // ---- softmax warps ----
        // P has kPBufs buffers: writing P of group i waits only for P V of group
        // i - kPBufs, which read the same buffer; a rescale of O waits for every earlier
        // P V. P V completions are waited for in order (pv_next: the first not yet
        // seen), so no barrier runs two phases ahead of these warps.
        const bool live = true;   // (spare softmax warps restore groups instead)
        bool ok = true;
        int pv_next = 0;
        auto pv_wait = [&](int upto) -> bool {   // P V of groups < upto completed
          while (pv_next < upto) {
            if (!wait_w(kPvDone + pv_next % kPBufs)) return false;
            ++pv_next;
          }
          tc_fence_after();
          return true;
        };
        for (int i = 0; i < ng; ++i) {
          const int s = i % kSlots;
          float z[32];
          float mx = -INFINITY;
          if (live) {
            S4KV_TRACE(tmark = global_ns();)
            if (!wait_w(kSFull + s)) { ok = false; break; }
            S4KV_TRACE({ const unsigned long long x = global_ns(); tq[1] += x - tmark; tmark = x; tq[4] += 1; tl(2 * tl_n); })
            tc_fence_after();
            uint32_t sr[32];
            tmem_ld32(tmem + t_row + 128 + kSCols * s, sr);
            tmem_wait_ld();
#pragma unroll
            for (int x = 0; x < 32; ++x) z[x] = __uint_as_float(sr[x]);
            if constexpr (BITS != 8) {   // plus the scores of the keys' low parts
              tmem_ld32(tmem + t_row + 128 + kSCols * s + kG, sr);
              tmem_wait_ld();
#pragma unroll
              for (int x = 0; x < 32; ++x) z[x] += __uint_as_float(sr[x]);
            }
            const int t0 = 32 * group_of(i);
            float mr = -INFINITY;   // maximum of the raw scores; zs > 0 keeps the order
            if (t0 + kG > free_end) {
#pragma unroll
              for (int x = 0; x < 32; ++x) {
                z[x] = t0 + x >= lim ? -INFINITY : z[x];
                mr = fmaxf(mr, z[x]);
              }
            } else {
#pragma unroll
              for (int x = 0; x < 32; ++x) mr = fmaxf(mr, z[x]);
            }
            mx = mr * zs;
          }
          S4KV_TRACE({ const unsigned long long x = global_ns(); tq[3] += x - tmark; tmark = x; })
          if (!pv_wait(i - kPBufs + 1)) { ok = false; break; }   // P buffer i % kPBufs is free
          S4KV_TRACE({ const unsigned long long x = global_ns(); tq[2] += x - tmark; tmark = x; })
          uint32_t pk[16];
#pragma unroll
          for (int x = 0; x < 16; ++x) pk[x] = 0u;
          if (live) {
            const bool need = mx > m_r + kLazy;
            if (__any_sync(0xffffffffu, need)) {
              const float mn = need ? mx : m_r;
              const float al = (!need || mn == -INFINITY) ? 1.0f : ex2(m_r - mn);
              m_r = mn;
              l_r *= al;
              if (i >= 1) {   // O must hold every earlier group before this column's row is rescaled
                if (!pv_wait(i)) { ok = false; break; }
#pragma unroll 1
                for (int ch = 0; ch < 4; ++ch) {
                  uint32_t orow[32];
                  tmem_ld32(tmem + t_row + 32 * ch, orow);
                  tmem_wait_ld();
#pragma unroll
                  for (int x = 0; x < 32; ++x) orow[x] = __float_as_uint(__uint_as_float(orow[x]) * al);
                  tmem_st32(tmem + t_row + 32 * ch, orow);
                }
                tmem_wait_st();
              }
            }
            // p = 2^(S zs - m), one FMA per score; a masked score (-inf) gives 0, and
            // while every score so far is masked (m = -inf) the offset is 0
            const float nm = m_r == -INFINITY ? 0.0f : -m_r;
            float sum = 0.0f;
#pragma unroll
            for (int x = 0; x < 32; x += 2) {
              const float p0 = ex2(fmaf(z[x], zs, nm));
              const float p1 = ex2(fmaf(z[x + 1], zs, nm));
              sum += p0 + p1;
              pk[x >> 1] = pack_f16x2(p0, p1);
            }
            l_r += sum;
          }
          if (live || i < kPBufs) {   // rows past the call's columns stay zero once every buffer is written
#pragma unroll
            for (int kg = 0; kg < 4; ++kg)
              *reinterpret_cast<uint4*>(base + kPo + (i % kPBufs) * kPTile + sw64_off(r, 8 * kg)) =
                  make_uint4(pk[4 * kg], pk[4 * kg + 1], pk[4 * kg + 2], pk[4 * kg + 3]);
          }
          fence_proxy_async();   // P's generic writes before the MMA reads them
          tc_fence_before();
          __syncwarp();
          if (lane == 0)
            asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(&bars[kPReady + i % kPBufs])) : "memory");
          S4KV_TRACE(tq[3] += global_ns() - tmark; tl(2 * tl_n + 1); ++tl_n;)
        }
        if (ok) pv_wait(ng);   // the last P V: O is final
      }
    }
    __syncthreads();   // every role has left its loop
    aborted = *flag != 0;
    if (aborted && warp == kLoadWarp && valid && ng > 0) {   // drain record copies still in flight
      if (lane == 0) report(a.status, S4KV_ERR_DEVICE_TIMEOUT, S4KV_DEV_TIMEOUT, b);
      // the copy of group j completes phase j / kRecStages of the barrier of stage j % kRecStages;
      // the last copy of stage s is of group j = s + kRecStages ((n_copies - 1 - s) / kRecStages)
      for (int s = 0; s < kRecStages && s < n_copies; ++s) {
        const int j = s + kRecStages * ((n_copies - 1 - s) / kRecStages);
        mbar_wait(&bars[kRecFull + s], static_cast<uint32_t>(j / kRecStages) & 1u, kDrainNs);
      }
      n_copies = 0;
    }
    if (tid == 0 && seg_start >= r0) {
      int ncon = 0;
      if (!own && slot_ok) ncon = owner_of(seg_end - 1, C, n_act) - gteam + 1;
      const long long first = 2LL * gteam + (seg_start <= r0 ? 0 : 1);
      meta_of(a)[static_cast<long long>(b) * a.H + h] =
          static_cast<long long>(static_cast<unsigned>(first)) | (static_cast<long long>(ncon) << 32);
    }
    if (warp < 4) {
      const bool have = valid && ng > 0 && !aborted;   // the same for every thread
      if (!have) {
        m_r = -INFINITY;
        l_r = 0.0f;
      }
      const float inv = (l_r > 0.0f ? 1.0f / l_r : 0.0f) * vsc;
      const int k = seg_start <= r0 ? 0 : 1;
      float* part = a.ws + (2LL * (static_cast<long long>(gteam) * kSlotWarps + r / 16) + k) * partial_floats(a.pcols);
#pragma unroll 1
      for (int ch = 0; ch < 4; ++ch) {
        uint32_t orow[32];
        if (have) {
          tmem_ld32(tmem + t_row + 32 * ch, orow);
          tmem_wait_ld();
        } else {
#pragma unroll
          for (int x = 0; x < 32; ++x) orow[x] = 0u;
        }
        if (r < cols) {
          if (own || !slot_ok) {
#pragma unroll
            for (int x = 0; x < 32; x += 4)
              store_out(a, row_of(r), (32 * ch + x) / 4,
                        make_float4(__uint_as_float(orow[x]) * inv, __uint_as_float(orow[x + 1]) * inv,
                                    __uint_as_float(orow[x + 2]) * inv, __uint_as_float(orow[x + 3]) * inv));
          } else {
#pragma unroll
            for (int x = 0; x < 32; x += 4)
              *reinterpret_cast<float4*>(part + (r % 16) * kD + 32 * ch + x) =
                  make_float4(__uint_as_float(orow[x]) * vsc, __uint_as_float(orow[x + 1]) * vsc,
                              __uint_as_float(orow[x + 2]) * vsc, __uint_as_float(orow[x + 3]) * vsc);
          }
        }
      }
      if (r < cols && !(own || !slot_ok)) {
        part[a.pcols * kD + 2 * (r % 16)] = m_r;
        part[a.pcols * kD + 2 * (r % 16) + 1] = l_r;
      }
    }
    if (tid == 0 && !aborted && valid && ng > 0) {   // nothing is in flight: fresh barriers for the next segment
      for (int k = 0; k < kNumBars; ++k) asm volatile("mbarrier.inval.shared::cta.b64 [%0];" ::"r"(smem_u32(&bars[k])) : "memory");
      init_bars();
    }
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    tc_fence_before();
    __syncthreads();   // O, Q, P and the slots are free for the next segment
    tc_fence_after();
    seg_start = seg_end;
    if (++h == a.H) {
      h = 0;
      if (++b >= a.B) break;
      sc = seg_cost<BITS>(a.seq_lens[b], a.R, a.tail_cost);
    }
  }
  S4KV_TRACE({
    if (lane == 0) {
      unsigned long long* out = reinterpret_cast<unsigned long long*>(meta_of(a) + meta_words(a.B, a.H)) +
                                (static_cast<long long>(blockIdx.x) * kSlotWarps + tslot) * kTraceWords;
      const unsigned long long t_end = global_ns();
      out[0] = t_end - tq[0];
      for (int k = 1; k < 5; ++k) out[k] = tq[k];
      out[5] = t_entry;   // absolute times: kernel entry, start of the segment loop, end
      out[6] = tq[0];
      out[7] = t_end;
    }
  })
  tc_fence_before();
  __syncthreads();
  if (warp == 0) asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "n"(kTmemCols));
  S4KV_TRACE(if (tid == 0) (reinterpret_cast<unsigned long long*>(meta_of(a) + meta_words(a.B, a.H)) +
                            static_cast<long long>(blockIdx.x) * kSlotWarps * kTraceWords)[8] = global_ns();)
}

// Merge for mq_kernel: one warp per (segment, column). Contributor i of a
// segment is team slot first + ... as in merge_kernel; the warp of column c in
// team t is warp (t / tpc) * kWarps + (t % tpc) * tw + c / 8 of the grid.
__global__ void __launch_bounds__(32 * kMergeWarps) mq_merge_kernel(DecodeArgs a) {
  asm volatile("griddepcontrol.wait;" ::: "memory");
  // tracing builds: the time this grid's first block passed the wait
  S4KV_TRACE(if (blockIdx.x == 0 && threadIdx.x == 0)
                 (reinterpret_cast<unsigned long long*>(meta_of(a) + meta_words(a.B, a.H)))[9] = global_ns();)
  constexpr int kWarps = S4KV_DECODE_WARPS;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const long long* desc = meta_of(a);
  const int cols = a.nq * a.g, tpc = kWarps / a.tw;
  const long long items = static_cast<long long>(a.B) * a.H * cols;
  const long long pf = partial_floats(a.pcols);
  for (long long it = static_cast<long long>(blockIdx.x) * kMergeWarps + warp; it < items;
       it += static_cast<long long>(gridDim.x) * kMergeWarps) {
    const int c = static_cast<int>(it % cols);
    const long long bh = it / cols;
    const long long d = __ldcg(desc + bh);
    const int nc = static_cast<int>(d >> 32);
    if (nc <= 0) continue;
    const long long first = static_cast<long long>(static_cast<unsigned>(d & 0xffffffffLL));
    const int tile = c / a.pcols, col = c % a.pcols;   // a warp holds pcols columns
    auto part = [&](int i) -> const float* {
      const long long ts = i == 0 ? first : (first & ~1LL) + 2LL * i;
      const long long gt = ts >> 1;
      const long long gwp = (gt / tpc) * kWarps + (gt % tpc) * a.tw + tile;
      return a.ws + (2LL * gwp + (ts & 1)) * pf;
    };
    float M = -INFINITY, L = 0.0f;
    float4 O = make_float4(0.0f, 0.0f, 0.0f, 0.0f);
    for (int i0 = 0; i0 < nc; i0 += kMC) {
      const int nch = min(kMC, nc - i0);
      const float* W = part(i0 + (lane < nch ? lane : 0)) + a.pcols * kD + 2 * col;
      const float mi = lane < nch ? __ldcg(W) : -INFINITY;
      const float li = lane < nch ? __ldcg(W + 1) : 0.0f;
      float4 r[kMC];
#pragma unroll
      for (int u = 0; u < kMC; ++u)
        r[u] = u < nch ? __ldcg(reinterpret_cast<const float4*>(part(i0 + u) + col * kD + 4 * lane))
                       : make_float4(0.0f, 0.0f, 0.0f, 0.0f);
      const float mn = fmaxf(M, warp_max(mi));
      const bool live = mn != -INFINITY;
      const float ao = live ? ex2(M - mn) : 1.0f;
      const float wi = live ? ex2(mi - mn) : 0.0f;
      L = fmaf(L, ao, warp_sum(wi * li));
      O = make_float4(O.x * ao, O.y * ao, O.z * ao, O.w * ao);
#pragma unroll
      for (int u = 0; u < kMC; ++u) {
        const float w = __shfl_sync(0xffffffffu, wi, u);
        O = make_float4(fmaf(w, r[u].x, O.x), fmaf(w, r[u].y, O.y), fmaf(w, r[u].z, O.z), fmaf(w, r[u].w, O.w));
      }
      M = mn;
    }
    const float inv = L > 0.0f ? 1.0f / L : 0.0f;
    const int b = static_cast<int>(bh / a.H), h = static_cast<int>(bh % a.H);
    store_out(a, (static_cast<long long>(b) * a.nq + c / a.g) * a.Hq + h * a.g + c % a.g, lane,
              make_float4(O.x * inv, O.y * inv, O.z * inv, O.w * inv));
  }
}

}  // namespace

size_t mq_timeline_bytes_per_warp() { return static_cast<size_t>(kMqTimelineWords) * 8; }

cudaError_t launch_mq(const DecodeArgs& args, int grid, cudaStream_t st) {
  static size_t attr[8] = {0, 0, 0, 0, 0, 0, 0, 0};
  DecodeArgs a = args;
  const int cols = a.nq * a.g;
  // KIVI pages: narrow calls fold the scales per warp (mq_kernel, 8 columns a warp);
  // from S4KV_MQ_TC_MIN_COLS_KIVI columns each group is restored once for tcgen05
  // (mqt_kernel); the mma.sync restore kernel (mqd_kernel, 16 columns a warp) when
  // chosen, or between the two thresholds if they are set apart.
  // FP8 pages: 16 columns a warp on mma.sync (mq_fp8_kernel), or, from
  // S4KV_MQ_TC_MIN_COLS columns or when chosen, each group widened once for tcgen05.
  const int choice = a.mq_kernel;
  const bool fp8 = a.bits == 8;
  const bool tc = choice == 3 || (choice == 0 && cols >= (fp8 ? S4KV_MQ_TC_MIN_COLS : S4KV_MQ_TC_MIN_COLS_KIVI));
  const bool restore = !fp8 && !tc && (choice == 2 || (choice == 0 && cols >= S4KV_MQ_RESTORE_MIN_COLS));
  a.pcols = fp8 || restore || tc ? 16 : 8;
  a.tw = (cols + a.pcols - 1) / a.pcols;
  if (restore && a.tw < kMqMinTeam) a.tw = kMqMinTeam;   // the team's regions hold a restored group
  if (tc) a.tw = S4KV_DECODE_WARPS;                       // one team per CTA
  // The restoring kernels' tail chunks (ring rows restored per token, the causal
  // mask) cost more against a main group than in decode. Their slices weigh a tail
  // chunk S4KV_MQT_TAIL_WEIGHT / 3 (tcgen05) and 5/3 (mma.sync restore) times the
  // decode weight: 5 and 5 for the default 3, the best of the weights measured on
  // Llama-3.1-8B shapes at nq = 8 and 16 (the tcgen05 kernel took 8 while its ring
  // rows were read one dependent load at a time).
  if (tc && !fp8) a.tail_cost = (S4KV_MQT_TAIL_WEIGHT * a.tail_cost + 1) / 3;
  else if (restore) a.tail_cost = (5 * a.tail_cost + 1) / 3;
  void (*kernel)(DecodeArgs) = fp8       ? (tc ? mqt_kernel<8> : mq_fp8_kernel)
                               : tc      ? (a.bits == 2 ? mqt_kernel<2> : mqt_kernel<4>)
                               : restore ? (a.bits == 2 ? mqd_kernel<2> : mqd_kernel<4>)
                                         : (a.bits == 2 ? mq_kernel<2> : mq_kernel<4>);
  const int which = fp8 ? (tc ? 7 : 0) : (tc ? 5 : restore ? 1 : 3) + (a.bits == 2 ? 1 : 0);
  const size_t smem = decode_smem_bytes(0, a.B);
  cudaError_t e = grant_smem(kernel, smem, &attr[which]);
  if (e != cudaSuccess) return e;
  kernel<<<grid, 32 * (tc ? mqt_warps(a.bits) : S4KV_DECODE_WARPS), smem, st>>>(a);
  e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  // The merge of a multi-query call has one item per (sequence, kv head, column): up to
  // S4KV_MQ_MERGE_BLOCKS merge blocks per attention CTA, so that the items' dependent loads
  // (descriptor, then partials) run side by side rather than one item after another per warp.
  const long long items = static_cast<long long>(a.B) * a.H * a.nq * a.g;
  if (items == 0) return cudaSuccess;
  e = prefer_max_shared(reinterpret_cast<const void*>(mq_merge_kernel));
  if (e != cudaSuccess) return e;
  long long blocks = (items + kMergeWarps - 1) / kMergeWarps;
  if (blocks > static_cast<long long>(S4KV_MQ_MERGE_BLOCKS) * grid) blocks = static_cast<long long>(S4KV_MQ_MERGE_BLOCKS) * grid;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>(blocks));
  cfg.blockDim = dim3(32 * kMergeWarps);
  cfg.dynamicSmemBytes = 0;
  cfg.stream = st;
  cudaLaunchAttribute attr_pdl[1];
  attr_pdl[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr_pdl[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr_pdl;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, mq_merge_kernel, a);
}

}  // namespace s4kv
