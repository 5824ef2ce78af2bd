// The attention kernel on CTA pairs (D = 128, every key visible: the dense,
// cross and prefix-cached forms).  Included once, by attn_fwd.cu, after
// attn_kernel.cuh, whose work schedule, softmax tile, merge and count-in it
// reuses.
//
// Why pairs.  With one CTA per SM, each 128-key step moves about 256 KB
// through shared memory: the S = Q K^T MMAs read Q and K (128 KB), the P V
// MMAs read V (64 KB), and TMA writes the next K and V tiles (64 KB).  At the
// tensor pipe's full rate that is all the shared-memory bandwidth there is,
// and the step settles well above its MMA time.  Two CTAs on an SM pair share
// each MMA (tcgen05 cta_group::2, M = 256): each supplies its own 128 query
// rows of A but only half of B, so each SM stores and reads half of every K
// tile (64 keys) and half of every V tile (64 head-dim columns): about 160 KB
// per step, and half the L2 traffic.
//
// Layout of one pair unit (b, h, 512 query rows from q0): pair tile i (i = 0,
// 1) is rows [q0 + 256 i, q0 + 256 i + 256); CTA r of the pair holds rows
// q0 + 256 i + 128 r .. + 127 of it, in its own tensor memory (S_i, O_i) and
// shared memory (Q_i).  The even CTA issues every MMA for both and commits to
// barriers in both; the odd CTA's MMA warp relays its loads' completions to
// the even CTA instead, so that each CTA's copies complete on its own
// barriers (and can be drained there after an abort).
#pragma once

#include "attn_kernel.cuh"

namespace ncp {

constexpr int PAIR_NSLOT = 8;            // half-tile ring slots (K halves and V halves alternate)
constexpr uint32_t HALF_BYTES = 16384;   // 64 keys x 128 dims, or 128 keys x 64 dims, bf16
constexpr uint32_t HALF_CHUNK = 8192;    // a K half: 64 rows x 128 bytes per 64-dim chunk

struct PairCfg {
  static constexpr int D = 128;
  static constexpr uint32_t TILE_BYTES = BM * D * 2;           // one 128-row Q tile
  static constexpr uint32_t CHUNK_BYTES = BM * 128;            // 128 rows x 128 bytes
  static constexpr uint32_t RING_OFF = 0;
  static constexpr uint32_t Q_OFF = RING_OFF + PAIR_NSLOT * HALF_BYTES;
  static constexpr uint32_t BAR_OFF = Q_OFF + 2 * TILE_BYTES;
  static constexpr uint32_t SMEM_BYTES = BAR_OFF + 1024 + 1024;  // control block + alignment slack
};

struct PairCtl {
  uint64_t q_full;                  // this CTA's Q tiles landed (its TMA)
  uint64_t q_free;                  // the item's last S MMAs are done (pair commit)
  uint64_t kv_full[PAIR_NSLOT];     // this CTA's half tile landed (its TMA)
  uint64_t kv_empty[PAIR_NSLOT];    // the MMAs reading the slot are done (pair commit)
  uint64_t s_full[2];               // S_i is complete (pair commit)
  uint64_t o_full[2];               // O_i is complete (pair commit)
  uint64_t p_full[2];               // even CTA: P_i written by the 8 softmax warps of the pair
  uint64_t o_free[2];               // even CTA: O_i read out by the 8 softmax warps of the pair
  uint64_t q_peer;                  // even CTA: the odd CTA's Q tiles landed (relayed)
  uint64_t kv_peer[PAIR_NSLOT];     // even CTA: the odd CTA's half tile landed (relayed)
  uint64_t part_done[2];
  uint64_t merge_ready[2];
  uint64_t drain;                   // abort: the pair's MMAs in flight are done
  int last[2];
  uint32_t tmem_base;
  int abort_flag;
};
static_assert(sizeof(PairCtl) <= 1024, "pair control block");

__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(PAIR_THREADS, 1)
    attn_pair_kernel(const __grid_constant__ Params p) {
  using C = PairCfg;
  constexpr int D = C::D;
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  // The pair's MMAs address both CTAs' operands at the same offsets: the
  // dynamic shared memory starts at the same address in every CTA.
  const uint32_t raw_u32 = smem_u32(smem_raw);
  const uint32_t base_u32 = (raw_u32 + 1023u) & ~1023u;
  uint8_t* base = smem_raw + (base_u32 - raw_u32);
  PairCtl* ctl = reinterpret_cast<PairCtl*>(base + C::BAR_OFF);
  volatile int* abort_flag = &ctl->abort_flag;

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const uint32_t rank = cluster_ctarank();          // 0: issues the MMAs
  const int pair = static_cast<int>(cluster_id_x());
  const int n_pairs = static_cast<int>(n_clusters_x());
  const int T0 = p.n_tiles[0];
  const int T = T0 + p.n_tiles[1];
  const uint64_t limit = p.wait_limit_ns;

  const uint32_t ring = base_u32 + C::RING_OFF;
  const uint32_t qs = base_u32 + C::Q_OFF;
  const uint32_t bar_q = smem_u32(&ctl->q_full);
  const uint32_t bar_qfree = smem_u32(&ctl->q_free);
  auto bar_kv_full = [&](int s) { return smem_u32(&ctl->kv_full[s]); };
  auto bar_kv_empty = [&](int s) { return smem_u32(&ctl->kv_empty[s]); };
  auto bar_kv_peer = [&](int s) { return smem_u32(&ctl->kv_peer[s]); };
  auto bar_s = [&](int i) { return smem_u32(&ctl->s_full[i]); };
  auto bar_p = [&](int i) { return smem_u32(&ctl->p_full[i]); };
  auto bar_o = [&](int i) { return smem_u32(&ctl->o_full[i]); };
  auto bar_ofree = [&](int i) { return smem_u32(&ctl->o_free[i]); };

  if (threadIdx.x == 0) {
    mbar_init(bar_q, 1);
    mbar_init(bar_qfree, 1);
    mbar_init(smem_u32(&ctl->q_peer), 1);
    for (int s = 0; s < PAIR_NSLOT; ++s) {
      mbar_init(bar_kv_full(s), 1);
      mbar_init(bar_kv_empty(s), 1);
      mbar_init(bar_kv_peer(s), 1);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(bar_s(i), 1);
      mbar_init(bar_o(i), 1);
      mbar_init(bar_p(i), 8);      // 4 softmax warps of each CTA
      mbar_init(bar_ofree(i), 8);  // 4 softmax warps of each CTA
      mbar_init(smem_u32(&ctl->part_done[i]), 4);
      mbar_init(smem_u32(&ctl->merge_ready[i]), 1);
    }
    mbar_init(smem_u32(&ctl->drain), 1);
    ctl->abort_flag = 0;
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
  }
  if (warp == MMA_WARP) {
    asm volatile("tcgen05.alloc.cta_group::2.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                     smem_u32(&ctl->tmem_base)),
                 "r"(TMEM_COLS)
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::2.sync.aligned;" ::: "memory");
  }
  tc_fence_before();
  cluster_sync();  // barriers initialised and tensor memory allocated in both CTAs
  tc_fence_after();
  const uint32_t tmem = ctl->tmem_base;

  // Loader bookkeeping for draining copies in flight after an abort.
  uint32_t ld_issued = 0, ld_parity = 0;
  int q_last = -1;
  const int g = n_pairs;
  const int c = pair;

  if (warp == PRODUCER_WARP) {
    // ------------------------------------------------------------ loader (both CTAs)
    // Whole warps run the loops of the loader, the relay and the MMA issuer,
    // converged; one elected lane issues each copy, MMA, commit and arrival.
    if (lane == 0) {
      prefetch_tmap(&p.tm_q);
      for (int s = 0; s < 2; ++s) {
        prefetch_tmap(&p.tm_kh[s]);
        prefetch_tmap(&p.tm_v[s]);
      }
    }
    __syncwarp();
    {
      int slot = 0;
      uint32_t phase = 0;
      bool ok = true;
      Item it;
      for (int n = 0; ok && schedule_item<false>(p.sc, T, g, c, n, it, nullptr); ++n) {
        const Unit& u = it.u;
        if (n > 0) {
          ok = warp_wait(bar_qfree, (n - 1) & 1, limit, abort_flag, 9);
          if (!ok) break;
        }
        const int nq_tiles = u.two ? 2 : 1;
        mbar_expect_tx_elect(bar_q, nq_tiles * C::TILE_BYTES);
        for (int i = 0; i < nq_tiles; ++i)
          for (int ch = 0; ch < 2; ++ch)
            tma_load_4d_elect(qs + i * C::TILE_BYTES + ch * C::CHUNK_BYTES, &p.tm_q, ch * 64, u.h,
                              u.q0 + 2 * BM * i + BM * static_cast<int>(rank), u.b, bar_q);
        q_last = n;
#pragma unroll 1
        for (int t = it.t_begin; t < it.t_end && ok; ++t) {
          const int seg = (t < T0) ? 0 : 1;
          const int tok0 = (t - (seg ? T0 : 0)) * BN;
          for (int kind = 0; kind < 2; ++kind) {
            ok = warp_wait(bar_kv_empty(slot), phase ^ 1u, limit, abort_flag, 1);
            if (!ok) break;
            const bool skip = (p.fault_mode == 1) && kind == 1 && t == 1 && n == 0 && c == 0 &&
                              rank == 0;
            if (!skip) {
              mbar_expect_tx_elect(bar_kv_full(slot), HALF_BYTES);
              const uint32_t dst = ring + slot * HALF_BYTES;
              if (kind == 0) {  // keys [tok0 + 64 r, + 64), both 64-dim chunks
                for (int ch = 0; ch < 2; ++ch)
                  tma_load_4d_elect(dst + ch * HALF_CHUNK, &p.tm_kh[seg], ch * 64, u.h,
                                    tok0 + 64 * static_cast<int>(rank), u.b, bar_kv_full(slot));
              } else {          // head-dim columns [64 r, + 64) of all 128 keys
                tma_load_4d_elect(dst, &p.tm_v[seg], 64 * static_cast<int>(rank), u.h, tok0, u.b,
                                  bar_kv_full(slot));
              }
              ld_issued |= 1u << slot;
              ld_parity = (ld_parity & ~(1u << slot)) | (phase << slot);
            }
            if (++slot == PAIR_NSLOT) {
              slot = 0;
              phase ^= 1u;
            }
          }
        }
      }
    }
    __syncwarp();
  } else if (warp == MMA_WARP && rank == 1) {
    // ------------------------------------- relay (odd CTA): its loads have landed
    {
      const uint32_t q_peer = map_to_rank(smem_u32(&ctl->q_peer), 0);
      int slot = 0;
      uint32_t phase = 0;
      bool ok = true;
      Item it;
      for (int n = 0; ok && schedule_item<false>(p.sc, T, g, c, n, it, nullptr); ++n) {
        ok = warp_wait(bar_q, n & 1, limit, abort_flag, 15);
        if (!ok) break;
        mbar_arrive_cluster_elect(q_peer);
#pragma unroll 1
        for (int t = it.t_begin; t < it.t_end && ok; ++t) {
          for (int kind = 0; kind < 2; ++kind) {
            ok = warp_wait(bar_kv_full(slot), phase, limit, abort_flag, 16);
            if (!ok) break;
            mbar_arrive_cluster_elect(map_to_rank(bar_kv_peer(slot), 0));
            if (++slot == PAIR_NSLOT) {
              slot = 0;
              phase ^= 1u;
            }
          }
        }
      }
    }
    __syncwarp();
  } else if (warp == MMA_WARP) {
    // ------------------------------------------------ MMA issuer (even CTA) for the pair
    {
      constexpr uint32_t IDESC_S = make_idesc(2 * BM, BN, false);
      constexpr uint32_t IDESC_PV = make_idesc(2 * BM, D, true);
      // S_i = Q_i K^T: A = this CTA's Q tile i (and the odd CTA's at the same
      // offset), B = the K half in slot k_slot (64 keys per CTA), 8 K-steps of 16.
      auto issue_s = [&](int i, int k_slot) {
        const uint32_t qa = qs + i * C::TILE_BYTES;
        const uint32_t kb = ring + k_slot * HALF_BYTES;
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) {
          const uint32_t a_off = (kk >> 2) * C::CHUNK_BYTES + (kk & 3) * 32;
          const uint32_t b_off = (kk >> 2) * HALF_CHUNK + (kk & 3) * 32;
          mma2_ss_elect(tmem + tmem_s_col(i), sw128_desc(qa + a_off, 16, 1024),
                        sw128_desc(kb + b_off, 16, 1024), IDESC_S, kk > 0);
        }
      };
      // O_i += P_i V: A = P_i in tensor memory, B = the V half in slot v_slot
      // (64 head-dim columns per CTA, MN-major), 8 K-steps of 16 keys.
      auto issue_pv = [&](int i, int v_slot, bool accumulate) {
        const uint32_t vb = ring + v_slot * HALF_BYTES;
#pragma unroll
        for (int kk = 0; kk < BN / 16; ++kk)
          mma2_ts_elect(tmem + tmem_o_col(i), tmem + tmem_s_col(i) + kk * 8,
                        sw128_desc(vb + kk * 16 * 128, C::CHUNK_BYTES, 1024), IDESC_PV,
                        (accumulate || kk > 0) ? 1u : 0u);
      };
      // Both CTAs' halves of the tile in `slot` have landed.
      auto kv_ready = [&](int slot, uint32_t ph, int site) -> bool {
        return warp_wait(bar_kv_full(slot), ph, limit, abort_flag, site) &&
               warp_wait_cluster(bar_kv_peer(slot), ph, limit, abort_flag, site);
      };
      int slot = 0;
      uint32_t phase = 0;
      uint32_t sc[2] = {0u, 0u};
      uint32_t oc[2] = {0u, 0u};
      bool ok = true;
      auto pv = [&](int i, int v_slot, bool accumulate) -> bool {
        if (!warp_wait_cluster(bar_p(i), (sc[i] - 1u) & 1u, limit, abort_flag, 4)) return false;
        if (!accumulate && oc[i] > 0 &&
            !warp_wait_cluster(bar_ofree(i), (oc[i] - 1u) & 1u, limit, abort_flag, 6))
          return false;
        tc_fence_after();
        issue_pv(i, v_slot, accumulate);
        return true;
      };
      Item it;
      for (int n = 0; ok && schedule_item<false>(p.sc, T, g, c, n, it, nullptr); ++n) {
        const int nq = it.u.two ? 2 : 1;
        ok = warp_wait(bar_q, n & 1, limit, abort_flag, 2) &&
             warp_wait_cluster(smem_u32(&ctl->q_peer), n & 1, limit, abort_flag, 2);
        if (!ok) break;
        int v_prev = -1;
        int j = 0;
#pragma unroll 1
        for (int t = it.t_begin; t < it.t_end && ok; ++t) {
          const int k_slot = slot;
          ok = kv_ready(k_slot, phase, 3);
          if (!ok) break;
          if (++slot == PAIR_NSLOT) { slot = 0; phase ^= 1u; }
          tc_fence_after();
#pragma unroll
          for (int i = 0; i < 2; ++i) {
            if (i >= nq || !ok) break;
            if (j > 0) {
              ok = pv(i, v_prev, j - 1 > 0);
              if (!ok) break;
            }
            issue_s(i, k_slot);
            mma2_commit_both_elect(bar_s(i));
            ++sc[i];
          }
          if (!ok) break;
          if (j > 0) mma2_commit_both_elect(bar_kv_empty(v_prev));
          mma2_commit_both_elect(bar_kv_empty(k_slot));
          const int v_slot = slot;
          ok = kv_ready(v_slot, phase, 5);
          if (!ok) break;
          if (++slot == PAIR_NSLOT) { slot = 0; phase ^= 1u; }
          v_prev = v_slot;
          ++j;
        }
        if (!ok) break;
        mma2_commit_both_elect(bar_qfree);
#pragma unroll
        for (int i = 0; i < 2; ++i) {
          if (i >= nq || !ok) break;
          ok = pv(i, v_prev, j - 1 > 0);
          if (!ok) break;
          mma2_commit_both_elect(bar_o(i));
          ++oc[i];
        }
        if (ok) mma2_commit_both_elect(bar_kv_empty(v_prev));
      }
    }
    __syncwarp();
  } else {
    // ------------------------------------------- softmax / correction / store (both CTAs)
    const int i = warp >> 2;
    const int wq = warp & 3;
    const uint32_t lane_base = static_cast<uint32_t>(wq * 32) << 16;
    const uint32_t s_addr = tmem + lane_base + tmem_s_col(i);
    const uint32_t o_addr = tmem + lane_base + tmem_o_col(i);
    const uint32_t p_full_even = map_to_rank(bar_p(i), 0);
    const uint32_t o_free_even = map_to_rank(bar_ofree(i), 0);
    const float sl2 = p.scale_log2;
    uint32_t sc = 0, oc = 0;
    bool ok = true;
    uint32_t mc = 0;
    const uint32_t bar_part = smem_u32(&ctl->part_done[i]);
    const uint32_t bar_merge = smem_u32(&ctl->merge_ready[i]);
    const int row = wq * 32 + lane;
    const uint32_t vis_all[4] = {~0u, ~0u, ~0u, ~0u};
    Item it;
    for (int n = 0; ok && schedule_item<false>(p.sc, T, g, c, n, it, nullptr); ++n) {
      const Unit& u = it.u;
      if (i == 1 && !u.two) continue;
      float m = -INFINITY;
      float l = 0.f;
      int j = 0;
#pragma unroll 1
      for (int t = it.t_begin; t < it.t_end; ++t) {
        ok = warp_wait(bar_s(i), sc & 1u, limit, abort_flag, 7);
        if (!ok) break;
        ++sc;
        tc_fence_after();
        const int seg = (t < T0) ? 0 : 1;
        const int valid = p.n_tok[seg] - (t - (seg ? T0 : 0)) * BN;
        softmax_tile<D, false>(s_addr, o_addr, valid, sl2, j > 0, vis_all, false, m, l);
        ++j;
        tmem_wait_st();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive_cluster(p_full_even);
      }
      if (!ok) break;
      ok = warp_wait(bar_o(i), oc & 1u, limit, abort_flag, 8);
      if (!ok) break;
      ++oc;
      tc_fence_after();
      uint32_t r[D];
#pragma unroll
      for (int cc = 0; cc < D; cc += 32) tmem_ld32(o_addr + cc, r + cc);
      tmem_wait_ld();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive_cluster(o_free_even);

      const int q = u.q0 + 2 * BM * i + BM * static_cast<int>(rank) + row;
      uint4* dst = reinterpret_cast<uint4*>(
          p.out + ((static_cast<size_t>(u.b) * p.Nq + q) * p.H + u.h) * D);
      if (it.tail >= 0) {
        // A piece of a tail unit: this CTA's partial rows go to its half of
        // the piece's slot (slot (slot0 + piece), CTA rank, tile i); the last
        // piece of this (unit, CTA, tile) to count in merges them.
        constexpr int NG = D / 4 + 1;
        auto part = [&](int k) {
          return reinterpret_cast<float4*>(p.ws_part) +
                 ((static_cast<size_t>(it.slot0 + k) * 2 + rank) * 2 + i) * NG * BM + row;
        };
        {
          float4* w = part(it.piece);
#pragma unroll
          for (int gg = 0; gg < D / 4; ++gg)
            __stcg(w + gg * BM, make_float4(__uint_as_float(r[4 * gg]), __uint_as_float(r[4 * gg + 1]),
                                            __uint_as_float(r[4 * gg + 2]),
                                            __uint_as_float(r[4 * gg + 3])));
          __stcg(w + (D / 4) * BM, make_float4(m, l, 0.f, 0.f));
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(bar_part);
        if (wq == 0) {
          ok = warp_wait(bar_part, mc & 1u, limit, abort_flag, 10);
          if (ok && lane == 0) {
            const int before =
                count_in(p.ws_count + (static_cast<size_t>(it.tail) * 2 + rank) * 2 + i, p.epoch);
            if (before < 0) {
              *abort_flag = 1;
              record_timeout(14);
            }
            ctl->last[i] = before == it.pieces - 1;
            mbar_arrive(bar_merge);
          }
          __syncwarp();
        }
        ok = warp_wait(bar_merge, mc & 1u, limit, abort_flag, 11);
        ++mc;
        if (!ok) break;
        if (!*reinterpret_cast<volatile int*>(&ctl->last[i])) continue;
        merge_pieces<D, 2>(part(0), it.pieces, q < p.Nq ? dst : nullptr);
        continue;
      }
      if (q < p.Nq) {
        const float inv_l = 1.f / l;
        const uint64_t inv2 = pk2(inv_l, inv_l);
#pragma unroll
        for (int cc = 0; cc < D; cc += 8) {
          uint32_t w[4];
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            float a0, a1;
            up2(fmul2(pk2(__uint_as_float(r[cc + 2 * e]), __uint_as_float(r[cc + 2 * e + 1])), inv2),
                a0, a1);
            w[e] = pack_bf16x2(a0, a1);
          }
          dst[cc / 8] = make_uint4(w[0], w[1], w[2], w[3]);
        }
      }
    }
  }

  // ------------------------------------------------------------------ exit
  tc_fence_before();
  __syncthreads();
  cluster_sync();
  const int pair_abort =
      *abort_flag | ld_shared_cluster(map_to_rank(smem_u32(&ctl->abort_flag), rank ^ 1u));
  if (pair_abort) {
    // Some role of the pair gave up: let this CTA's copies and the pair's MMAs
    // in flight land before the tensor memory is released (bounded waits).
    if (warp == PRODUCER_WARP && lane == 0) {
      if (q_last >= 0) wait_drain(bar_q, q_last & 1, limit);
      for (int s = 0; s < PAIR_NSLOT; ++s)
        if (ld_issued & (1u << s)) wait_drain(bar_kv_full(s), (ld_parity >> s) & 1u, limit);
    }
    if (warp == MMA_WARP) {
      // The even CTA's MMAs were issued by its elected lane: commit from it too.
      if (rank == 0) mma2_commit_both_elect(smem_u32(&ctl->drain));
      if (lane == 0) wait_drain(smem_u32(&ctl->drain), 0, limit);
    }
    __syncwarp();
  }
  tc_fence_before();
  __syncthreads();
  cluster_sync();
  if (warp == MMA_WARP) {
    tc_fence_after();
    asm volatile("tcgen05.dealloc.cta_group::2.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(TMEM_COLS)
                 : "memory");
  }
}

}  // namespace ncp
