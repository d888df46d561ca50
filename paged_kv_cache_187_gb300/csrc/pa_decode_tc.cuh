// pa_decode_tc.cuh -- multi-query paged decode on the 5th-generation tensor cores
// (tcgen05, tensor memory), head_size 128.
//
// What it computes: the multi-query decode of pa_decode.cuh ("vLLM Project Update" talk,
// speculative-decoding part: attention for several query tokens per sequence): for every
// (sequence s, query token j, query head h) row,
//     out = sum_t softmax_t(scale * q . k_t) v_t  over t < L - q_len + j + 1,
// K/V paged through the block table, kv head h / group.
//
// With many query rows per kv head (q_len x group >= 16) the decode is a real contraction:
// a 128-token tile against up to 32 rows costs 2 x 128 x 32 x 128 multiply-adds per K/V
// byte pair, more than mma.sync sustains at the warps per SM its registers allow.  Here
// the contraction runs on tcgen05 with the accumulators in tensor memory:
//   * tile = 128 tokens (128 / block_size paged blocks), gathered by TMA into a K ring and
//     a V ring of 128-byte-swizzled [2 halves][128 tokens][128 B] stages;
//   * S^T = K Q^T:  M = 128 tokens, N = RPAD (16 or 32) query rows, K = 128 head dims;
//     A = the K tile (K-major), B = Q (K-major, staged swizzled by the producer);
//   * softmax over the tile's tokens: 4 warps, one tensor-memory lane (token) per thread,
//     against a per-row reference that moves only when a score passes it (one vote of
//     the four warps per tile; column maxima by a transposed warp reduction and a
//     cross-warp exchange only when it moves);
//   * O^T += V^T P^T:  M = 128 head dims, N = RPAD, K = 128 tokens; A = the V tile
//     (MN-major), B = P^T (MN-major: each softmax thread writes its token's row of
//     weights, as P_hi + P_lo for bf16, in 16-byte stores);
//     O^T stays in tensor memory and is rescaled there when a row's reference moves.
// Roles, three warpgroups: warps 0-3 run the softmax; warps 4-7 the epilogue of each unit
// (O^T out of tensor memory, normalisation, stores, the partition merge), double-buffered
// in tensor memory so that the next unit's softmax never waits for it; warp 8 streams K
// tiles (TMA), warp 9 issues the MMAs (one thread), warp 10 streams V tiles.  The softmax
// warpgroup takes most of the register file (setmaxnreg).  Work units are the same
// (sequence, kv head, partition, row chunk) units as the other decode kernels, claimed
// from the same plan; partitions are multiples of 128 tokens.  Every wait is bounded; the
// softmax warps, and the epilogue warps, take each abort decision together so that none
// is left at a named barrier.
#pragma once

#include "pa_decode.cuh"

namespace pa {
namespace tc {

constexpr int kTok = 128;              // tokens per tile
constexpr int kD = 128;                // head size
constexpr uint32_t kHalf = kTok * 128; // one 64-column half of a 128-row tile, bytes
constexpr int kSoftThreads = 128;      // the four softmax warps
constexpr int kEpiThreads = 128;       // the four epilogue warps
constexpr int kBarSoft = 1;            // named barrier of the softmax warps
constexpr int kBarEpi = 2;             // named barrier of the epilogue warps
// Warp roles (one warpgroup each for the softmax and the epilogue, then the single warps)
constexpr int kWarpEpi0 = 4, kWarpK = 8, kWarpMma = 9, kWarpV = 10;
constexpr float kSlack = 8.f;          // a moved reference sits this far above the largest score

template <bool BF16_, int BS_, int RPAD_>
struct TcCfg {
    static constexpr bool kBf16 = BF16_;
    static constexpr int BS = BS_;
    static constexpr int RPAD = RPAD_;            // query rows per unit: N of both MMAs
    static constexpr int BLOCKS = kTok / BS_;     // paged blocks per tile
    // K and V ring stages.  The kernel streams at the rate the bytes in flight allow, so
    // both rings take 3 stages (192 KB) whatever the rows per unit; a K tile starts each
    // tile's chain (QK^T, softmax, PV), so K never gets fewer stages than V.
    static constexpr int NK = 3, NV = 3;
    static constexpr int NQ = 2;                  // unit descriptor slots
    // P as hi + lo bf16 terms, or one fp16 term.  The terms are stacked along N (entries
    // n and RPAD + n of a token's P^T row), so one PV instruction per k-step reads the V
    // tile once and accumulates O_hi and O_lo side by side; the epilogue adds them.
    static constexpr int PSPLIT = BF16_ ? 2 : 1;
    static constexpr int NPV = PSPLIT * RPAD_;           // N of the PV product
    static constexpr uint32_t TILE_BYTES = 2 * kHalf;   // K (or V) of one tile: 32 KB
    static constexpr uint32_t QHALF = RPAD_ * 128;      // one 64-dim half of Q
    // P^T, the PV's B operand, MN-major: token t's NPV entries (rows n, then the second
    // term's) fill one PROW-byte row, written by t's softmax thread in 16-byte chunks; the
    // chunks are swizzled within atoms of 8 rows (128-, 64- or 32-byte swizzle: one MMA's
    // N entries never cross an atom)
    static constexpr uint32_t PROW = NPV * 2;           // 128, 64 or 32 bytes per token
    static constexpr uint32_t PBUF = kTok * PROW;       // one tile's P^T
    // Q buffers (units) and P^T buffers (tiles): two where shared memory allows, so that
    // the next unit's Q, or the next tile's P^T, is written while the MMAs read the
    // current one.  With 32 rows they make room for the rings: one Q buffer (the next
    // unit's Q waits for the current unit's last QK^T), and for bf16 (P^T in two terms)
    // one P^T buffer (the next tile's P^T waits for the current PV).
    static constexpr int NQB = RPAD_ == 16 ? 2 : 1;
    static constexpr int NP = (RPAD_ == 32 && BF16_) ? 1 : 2;
    // warps: 0-3 softmax, 4-7 epilogue, 8 K producer (claims units, stages Q), 9 MMA
    // issuer, 10 V producer, 11 idle (it completes the third warpgroup)
    static constexpr int THREADS = 12 * 32;
    // Registers per thread: the launch gives every thread REG_LAUNCH (65536 / 384, rounded
    // down to a multiple of 8); the epilogue and the single-warp roles hand part of theirs
    // to the softmax warps.  The increase must be covered by the decreases.
    static constexpr int REG_LAUNCH = 168, REG_SOFT = 232, REG_EPI = 128, REG_AUX = 144;
    static_assert(REG_SOFT + REG_EPI + REG_AUX <= 3 * REG_LAUNCH, "register split");
    static_assert(REG_LAUNCH * THREADS <= 65536, "register file");
    // tensor memory: S^T double-buffered (2 x RPAD columns), then O^T of two consecutive
    // units (2 x NPV columns)
    static constexpr uint32_t COL_S = 0, COL_O = 2 * RPAD_;
    static constexpr uint32_t TMEM_NEED = COL_O + 2 * NPV;
    static constexpr uint32_t TMEM_COLS = TMEM_NEED <= 64 ? 64 : TMEM_NEED <= 128 ? 128 : 256;
    static_assert(RPAD_ == 16 || RPAD_ == 32, "rows per unit");
    static_assert(BS_ == 16 || BS_ == 32, "block size");
};

template <class C>
struct alignas(1024) TcSmem {
    uint8_t k[C::NK][C::TILE_BYTES];
    uint8_t v[C::NV][C::TILE_BYTES];
    uint8_t q[C::NQB][2 * C::QHALF];         // Q of consecutive units
    uint8_t p[C::NP][C::PBUF];               // P^T of consecutive tiles
    alignas(16) float red[2][C::RPAD][4];   // per-warp column maxima, by tile parity
    // A finished unit handed from the softmax to the epilogue warps, by unit parity: the
    // per-warp column exp-sums, the row references and the descriptor
    alignas(16) float lred[2][C::RPAD][4];
    alignas(16) float mrow[2][C::RPAD];
    UnitDesc eunit[2];
    alignas(16) uint16_t ostage[16][kD];     // 16 output rows on their way out
    uint64_t k_full[C::NK], k_empty[C::NK], v_full[C::NV], v_empty[C::NV];
    uint64_t s_full[2], p_full[2], pv_done[2];
    uint64_t q_full[2], q_empty[2], drain;
    // o_full[b]: the last PV of the unit in O^T buffer b has completed; o_empty[b]: the
    // epilogue warps have read that buffer (and the hand-over slot of the same parity);
    // e_full[b]: the softmax warps have filled hand-over slot b
    uint64_t o_full[2], o_empty[2], e_full[2];
    uint64_t u_full[C::NQ], u_empty[C::NQ];
    UnitDesc unit[C::NQ];
    uint32_t k_issued[C::NK], v_issued[C::NV];   // TMA tiles issued per stage (producer)
    uint32_t k_done[C::NK], v_done[C::NV];       // ... whose MMAs were issued (MMA thread)
    uint32_t tmem_base;
    int32_t last_flag;
    volatile int32_t abort;
};

template <class C>
constexpr size_t tc_smem_bytes() {
    return sizeof(TcSmem<C>) + 1024;
}

// Lane l ends with the max (sum) over the warp of column l % R of v[0..R).
template <int R, bool kMax>
__device__ __forceinline__ float warp_transpose_reduce(float (&v)[R], int lane) {
    auto op = [](float a, float b) { return kMax ? fmaxf(a, b) : a + b; };
    int w = R;
#pragma unroll
    for (int s = R / 2; s >= 1; s >>= 1) {
        const bool up = (lane & s) != 0;
#pragma unroll
        for (int i = 0; i < R / 2; ++i) {
            if (i < w / 2) {
                const float send = up ? v[i] : v[i + w / 2];
                const float keep = up ? v[i + w / 2] : v[i];
                v[i] = op(keep, __shfl_xor_sync(0xffffffffu, send, s));
            }
        }
        w >>= 1;
    }
    float r = v[0];
#pragma unroll
    for (int s = R; s < 32; s <<= 1) r = op(r, __shfl_xor_sync(0xffffffffu, r, s));
    return r;
}

// Row of `out` / q for query row r of a unit: (query token r / group, head kvh*group + r % group).
__device__ __forceinline__ size_t mq_out_row(const DecodeParams& p, int32_t seq, int32_t kvh, int r) {
    const int j = r / p.group;
    return ((size_t)seq * p.q_len + j) * p.num_q_heads + (size_t)kvh * p.group + (r - j * p.group);
}

template <class C>
__global__ void __launch_bounds__(C::THREADS, 1)
    paged_decode_tc_kernel(const __grid_constant__ CUtensorMap kmap,
                           const __grid_constant__ CUtensorMap vmap, const DecodeParams p,
                           const int32_t persistent, const int32_t num_units_v1) {
    extern __shared__ uint8_t smem_raw[];
    TcSmem<C>& sm = *reinterpret_cast<TcSmem<C>*>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    constexpr int RPAD = C::RPAD;

    if (threadIdx.x == 0) {
        for (int i = 0; i < C::NK; ++i) {
            mbar_init(&sm.k_full[i], 1);
            mbar_init(&sm.k_empty[i], 1);
            sm.k_issued[i] = sm.k_done[i] = 0;
        }
        for (int i = 0; i < C::NV; ++i) {
            mbar_init(&sm.v_full[i], 1);
            mbar_init(&sm.v_empty[i], 1);
            sm.v_issued[i] = sm.v_done[i] = 0;
        }
        for (int i = 0; i < 2; ++i) {
            mbar_init(&sm.s_full[i], 1);
            mbar_init(&sm.p_full[i], 4);
            mbar_init(&sm.pv_done[i], 1);
        }
        for (int i = 0; i < 2; ++i) {
            mbar_init(&sm.q_full[i], 1);
            mbar_init(&sm.q_empty[i], 1);
            mbar_init(&sm.o_full[i], 1);
            mbar_init(&sm.o_empty[i], 4);   // the four epilogue warps
            mbar_init(&sm.e_full[i], 4);    // the four softmax warps
        }
        mbar_init(&sm.drain, 1);
        for (int i = 0; i < C::NQ; ++i) {
            mbar_init(&sm.u_full[i], 1);
            mbar_init(&sm.u_empty[i], 6);   // MMA thread, 4 softmax warps, V producer
        }
        sm.abort = 0;
        fence_barrier_init();
        prefetch_tensor_map(&kmap);
        prefetch_tensor_map(&vmap);
    }
    if (warp == kWarpMma) {
        tmem_alloc(&sm.tmem_base, C::TMEM_COLS);
        tmem_relinquish();
    }
    tmem_fence_before_sync();
    __syncthreads();
    tmem_fence_after_sync();
    const uint32_t tmem = sm.tmem_base;
    grid_dependency_wait();   // the plan / reshape kernel before this one has finished

    const int32_t Hkv = p.num_kv_heads, RC = p.row_chunks, upl = Hkv * RC;
    // Producers (K and V warps, all lanes): block-table entries first .. first+31 of a
    // unit's sequence, one per lane; entries at or past `end`, or outside the pool, become a
    // row past the tensor map (TMA reads zeros there).
    auto load_chunk = [&](const UnitDesc& u, int32_t first, int32_t end) {
        int32_t phys = p.num_blocks;
        if (first + lane < end) {
            phys = p.block_tables[(size_t)u.seq * p.max_blocks_per_seq + first + lane];
            if (phys < 0 || phys >= p.num_blocks) {
                if (u.kvh == 0 && u.row0 == 0) flag_error(p.status, PA_DEVERR_BAD_BLOCK_);
                phys = p.num_blocks;
            }
        }
        return phys;
    };
    // Producers: one tile (BLOCKS paged blocks, both 64-column halves) into stage n % ns of
    // a ring; block b's entry sits in lane within + b of `chunk`.  Lane 0 posts the expected
    // bytes, then lane 2b + h copies half h of block b.  False when the wait gave up.
    auto issue_tile = [&](uint8_t (*ring)[C::TILE_BYTES], uint64_t* full, uint64_t* empty,
                          uint32_t* issued, uint32_t ns, uint32_t n, const CUtensorMap* map,
                          int32_t chunk, int32_t within, int32_t kvh) {
        const uint32_t st = n % ns, ph = ((n / ns) & 1) ^ 1;
        bool ok = true;
        if (lane == 0) {
            ok = mbar_wait(&empty[st], ph);
            if (ok) {
                mbar_arrive_expect_tx(&full[st], C::TILE_BYTES);
                issued[st] += 1;
            }
        }
        ok = __shfl_sync(0xffffffffu, ok ? 1 : 0, 0) != 0;
        if (!ok) return false;
        __syncwarp();   // the expected bytes are posted before any copy is issued
        const int b = (lane >> 1) & (C::BLOCKS - 1), h = lane & 1;
        const int32_t pb = __shfl_sync(0xffffffffu, chunk, within + b);
        if (lane < 2 * C::BLOCKS) {
            const int32_t y = (pb * Hkv + kvh) * C::BS;
            tma_load_2d(ring[st] + h * kHalf + b * C::BS * 128, map, h * 64, y, &full[st],
                        l2_evict_first_policy());
        }
        return true;
    };

    if (warp >= kWarpK) {
        // the single-warp roles (and the idle warp) hand registers to the softmax warps;
        // the whole warpgroup releases them together, before it splits into roles
        warpgroup_reg_release<C::REG_AUX>();
        if (warp == kWarpK) {
            // ------------------------------------------------------------ K producer
            const int32_t total = persistent ? (int32_t)p.hdr->total_units : num_units_v1;
            const int32_t P = persistent ? (int32_t)p.hdr->partition_size : 0;
            const int4 kNoEntry = make_int4(0, 0, 0, 0);
            // Unit w as a descriptor: V1 units from the grid index, V2 units from the plan's
            // list entry e (sequence, partition, first partition slot, length).
            auto describe = [&](int32_t w, int4 e) {
                UnitDesc u;
                u.seq = -1;
                u.kvh = u.tok0 = u.tok1 = u.pbase = u.row0 = u.nrows = u.len = 0;
                u.pslot = -1;
                u.nparts = 1;
                u.pad[0] = u.pad[1] = 0;
                if (w < total) {
                    const int32_t wu = w / RC;
                    u.row0 = (w - wu * RC) * RPAD;
                    u.nrows = min(RPAD, p.rows - u.row0);
                    u.kvh = wu % Hkv;
                    if (!persistent) {
                        u.seq = wu / Hkv;
                        u.tok1 = clamped_len(p, u.seq, u.kvh == 0 && u.row0 == 0);
                        u.len = u.tok1;
                    } else {
                        u.seq = e.x;
                        u.tok0 = e.y * P;
                        u.tok1 = min(u.tok0 + P, e.w);
                        u.nparts = e.w > 0 ? (e.w + P - 1) / P : 1;
                        u.pbase = e.z;
                        u.pslot = u.nparts > 1 ? e.z + e.y : -1;
                        u.len = e.w;
                    }
                }
                return u;
            };
            // The next unit is claimed as soon as the current one is published and its list
            // entry is read after the current unit's first tile, so neither round trip stalls
            // the tile stream.
            // every CTA starts with the unit of its own index; later units are claimed from the
            // counter, past the first gridDim.x
            int32_t w = (int32_t)blockIdx.x;
            int4 e = (persistent && w < total) ? p.part_list[w / upl] : kNoEntry;
            uint32_t kt = 0;   // tiles issued into the K ring
            bool ok = true;
            for (uint32_t it = 0; ok; ++it) {
                const bool done = w >= total || warp_sees_abort(sm.abort);
                const UnitDesc u = describe(done ? total : w, e);
                const uint32_t qs = it % C::NQ, qph = ((it / C::NQ) & 1) ^ 1;
                if (lane == 0) {
                    ok = mbar_wait(&sm.u_empty[qs], qph);
                    if (ok) {
                        sm.unit[qs] = u;
                        mbar_arrive(&sm.u_full[qs]);
                    }
                }
                ok = __shfl_sync(0xffffffffu, ok ? 1 : 0, 0) != 0;
                // every K tile of this CTA is issued: the kernels queued after this one may
                // launch once all CTAs are here (each waits for this kernel before it touches
                // what this one uses)
                if (ok && u.seq < 0 && PA_DECODE_TRIGGER && lane == 0) allow_dependent_launch();
                if (!ok || u.seq < 0) break;
                // Q rows of the unit, staged into its Q buffer (unit parity) in the 128B-swizzled
                // K-major layout, rows past the unit's zero: loads now, stores after the first
                // tile's copies are issued.  The buffer's previous unit has finished its QK^T.
                constexpr int kQChunks = RPAD * 16 / 32;   // 16-byte chunks per lane
                uint4 qv[kQChunks];
    #pragma unroll
                for (int i = 0; i < kQChunks; ++i) {
                    const int c = lane + 32 * i, n = c >> 4;
                    qv[i] = make_uint4(0u, 0u, 0u, 0u);
                    if (n < u.nrows)
                        qv[i] = __ldg(reinterpret_cast<const uint4*>(
                                          reinterpret_cast<const uint16_t*>(p.q) +
                                          mq_out_row(p, u.seq, u.kvh, u.row0 + n) * kD) + (c & 15));
                }
                bool q_staged = false;
                auto stage_q = [&]() {
                    const uint32_t qb = it % C::NQB;
                    if (lane == 0) ok = mbar_wait(&sm.q_empty[qb], ((it / C::NQB) & 1) ^ 1);
                    ok = __shfl_sync(0xffffffffu, ok ? 1 : 0, 0) != 0;
                    if (ok) {
    #pragma unroll
                        for (int i = 0; i < kQChunks; ++i) {
                            const int c = lane + 32 * i, n = c >> 4, ch = c & 15, h = ch >> 3, cc = ch & 7;
                            *reinterpret_cast<uint4*>(sm.q[qb] + h * C::QHALF + n * 128 + ((cc ^ (n & 7)) << 4)) = qv[i];
                        }
                        fence_proxy_async_smem();
                        __syncwarp();
                        if (lane == 0) mbar_arrive(&sm.q_full[qb]);
                    }
                    q_staged = true;
                };
                int32_t claimed = total;
                if (persistent && lane == 0) claimed = (int32_t)(gridDim.x + atomicAdd(&p.hdr->counter, 1u));
                int32_t w_next = total;
                int4 e_next = kNoEntry;
                bool have_next = false;
                auto fetch_next = [&]() {
                    w_next = persistent ? __shfl_sync(0xffffffffu, claimed, 0) : total;
                    e_next = (persistent && w_next < total) ? p.part_list[w_next / upl] : kNoEntry;
                    have_next = true;
                };
                const int32_t nb0 = u.tok0 / C::BS, nb1 = (u.tok1 + C::BS - 1) / C::BS;
                const int32_t ntiles = (u.tok1 - u.tok0 + kTok - 1) / kTok;
                // block-table chunks of 32 entries, the next one always in flight
                int32_t chunk = 0;
                int32_t cur = load_chunk(u, nb0, nb1), nxt = load_chunk(u, nb0 + 32, nb1);
                for (int32_t j = 0; j < ntiles && ok; ++j) {
                    const int32_t tb = j * C::BLOCKS;    // first block of the tile in the unit
                    if ((tb >> 5) != chunk) {
                        chunk = tb >> 5;
                        cur = nxt;
                        nxt = load_chunk(u, nb0 + 32 * (chunk + 1), nb1);
                    }
                    ok = issue_tile(sm.k, sm.k_full, sm.k_empty, sm.k_issued, C::NK, kt, &kmap, cur,
                                    tb & 31, u.kvh);
                    ++kt;
                    if (j == 0) {
                        stage_q();
                        fetch_next();
                    }
                }
                if (ok && !q_staged) stage_q();
                if (!have_next) fetch_next();
                w = w_next;
                e = e_next;
            }
            if (!ok && lane == 0) {
                flag_error(p.status, PA_DEVERR_TIMEOUT_);
                sm.abort = 1;
            }
        } else if (warp == kWarpV) {
            // ------------------------------------------------------------ V producer
            // Follows the units the K producer publishes and streams their V tiles into the V
            // ring, so that a V stage still held by a PV never delays the next K tile.
            uint32_t vt = 0;
            bool ok = true;
            for (uint32_t it = 0; ok; ++it) {
                const uint32_t qs = it % C::NQ;
                ok = mbar_wait_warp(&sm.u_full[qs], (it / C::NQ) & 1);
                if (!ok) break;
                const UnitDesc u = sm.unit[qs];
                __syncwarp();
                if (lane == 0) mbar_arrive(&sm.u_empty[qs]);
                if (u.seq < 0) break;
                const int32_t nb0 = u.tok0 / C::BS, nb1 = (u.tok1 + C::BS - 1) / C::BS;
                const int32_t ntiles = (u.tok1 - u.tok0 + kTok - 1) / kTok;
                int32_t chunk = 0;
                int32_t cur = load_chunk(u, nb0, nb1), nxt = load_chunk(u, nb0 + 32, nb1);
                for (int32_t j = 0; j < ntiles && ok; ++j) {
                    const int32_t tb = j * C::BLOCKS;
                    if ((tb >> 5) != chunk) {
                        chunk = tb >> 5;
                        cur = nxt;
                        nxt = load_chunk(u, nb0 + 32 * (chunk + 1), nb1);
                    }
                    ok = issue_tile(sm.v, sm.v_full, sm.v_empty, sm.v_issued, C::NV, vt, &vmap, cur,
                                    tb & 31, u.kvh);
                    ++vt;
                }
            }
            if (!ok && lane == 0) {
                flag_error(p.status, PA_DEVERR_TIMEOUT_);
                sm.abort = 1;
            }
        } else if (warp == kWarpMma) {
            // ------------------------------------------------------------ MMA issuer
            if (lane == 0) {
                constexpr uint32_t kIdQK = mma_idesc_f16(C::kBf16, 0, 0, kTok, RPAD);
                constexpr uint32_t kIdPV = mma_idesc_f16(C::kBf16, 1, 1, kD, C::NPV);
                uint32_t kt = 0, vt = 0, gt = 0, un = 0;
                bool ok = true;
                // P^T V of tile t (global tile index), into O^T buffer un & 1.  The first PV of
                // a unit waits until the epilogue warps have read that buffer's previous unit.
                auto pv = [&](uint32_t t, bool first) {
                    const uint32_t b = t & 1;
                    ok = mbar_wait(&sm.p_full[b], (t >> 1) & 1);
                    if (ok && first) ok = mbar_wait(&sm.o_empty[un & 1], ((un >> 1) & 1) ^ 1);
                    const uint32_t vs = vt % C::NV;
                    if (ok) ok = mbar_wait(&sm.v_full[vs], (vt / C::NV) & 1);
                    if (!ok) return;
                    tmem_fence_after_sync();
                    // descriptors differ from the stage's base only in the start address
                    // (16-byte units, low bits): built once, offset per k-step
                    const uint64_t va = smem_desc_sw128(smem_u32(sm.v[vs]), kHalf, 1024);
                    const uint64_t pb = smem_desc(smem_u32(sm.p[t % C::NP]), C::PBUF, 8 * C::PROW, C::PROW);
    #pragma unroll
                    for (int i = 0; i < kTok / 16; ++i)
                        mma_f16_ss(tmem + C::COL_O + (un & 1) * C::NPV, va + (uint64_t)(i * (2048 >> 4)),
                                   pb + (uint64_t)((i * 16 * C::PROW) >> 4), kIdPV,
                                   !(first && i == 0));
                    mma_commit(&sm.v_empty[vs]);
                    mma_commit(&sm.pv_done[b]);
                    sm.v_done[vs] += 1;
                    ++vt;
                };
                for (uint32_t it = 0; ok; ++it) {
                    const uint32_t qs = it % C::NQ;
                    ok = mbar_wait(&sm.u_full[qs], (it / C::NQ) & 1);
                    if (!ok) break;
                    const UnitDesc u = sm.unit[qs];
                    mbar_arrive(&sm.u_empty[qs]);
                    if (u.seq < 0) break;
                    ok = mbar_wait(&sm.q_full[un % C::NQB], (un / C::NQB) & 1);
                    if (!ok) break;
                    const uint64_t qd = smem_desc_sw128(smem_u32(sm.q[un % C::NQB]), 16, 1024);
                    const int32_t ntiles = (u.tok1 - u.tok0 + kTok - 1) / kTok;
                    for (int32_t j = 0; j < ntiles && ok; ++j) {
                        // this tile's QK^T and the previous tile's PV, in whichever order their
                        // inputs (K tile; published P^T) arrive
                        bool pv_prev = j > 0;
                        const uint32_t ks = kt % C::NK;
                        const uint32_t kbar = smem_u32(&sm.k_full[ks]), kph = (kt / C::NK) & 1;
                        const uint64_t t0 = global_timer_ns();
                        while (pv_prev && !mbar_try_wait(kbar, kph)) {
                            if (mbar_try_wait(smem_u32(&sm.p_full[(gt - 1) & 1]), ((gt - 1) >> 1) & 1)) {
                                pv(gt - 1, j == 1);
                                pv_prev = false;
                            } else if (global_timer_ns() - t0 > kWaitLimitNs) {
                                ok = false;
                            }
                            if (!ok) break;
                        }
                        if (!ok) break;
                        ok = mbar_wait(&sm.k_full[ks], kph);
                        if (!ok) break;
                        tmem_fence_after_sync();
                        const uint64_t ka = smem_desc_sw128(smem_u32(sm.k[ks]), 16, 1024);
                        const uint32_t d = tmem + C::COL_S + (gt & 1) * RPAD;
    #pragma unroll
                        for (int i = 0; i < kD / 16; ++i)
                            mma_f16_ss(d, ka + (uint64_t)(((i >> 2) * kHalf + (i & 3) * 32) >> 4),
                                       qd + (uint64_t)(((i >> 2) * C::QHALF + (i & 3) * 32) >> 4), kIdQK,
                                       i > 0);
                        mma_commit(&sm.s_full[gt & 1]);
                        mma_commit(&sm.k_empty[ks]);
                        sm.k_done[ks] += 1;
                        ++kt;
                        if (pv_prev) pv(gt - 1, j == 1);
                        ++gt;
                    }
                    mma_commit(&sm.q_empty[un % C::NQB]);   // this unit's QK^T are all issued
                    if (ok && ntiles > 0) pv(gt - 1, ntiles == 1);
                    // a unit without tiles issues no PV but still takes its O^T buffer in
                    // turn, so that o_full never runs two phases ahead of the epilogue
                    else if (ok) ok = mbar_wait(&sm.o_empty[un & 1], ((un >> 1) & 1) ^ 1);
                    if (!ok) break;
                    mma_commit(&sm.o_full[un & 1]);
                    ++un;
                }
                if (!ok) {
                    flag_error(p.status, PA_DEVERR_TIMEOUT_);
                    sm.abort = 1;
                }
                // every MMA this thread issued has completed before tensor memory is freed
                mma_commit(&sm.drain);
                (void)mbar_wait(&sm.drain, 0);
            }
            __syncwarp();
        }
    } else if (warp < kWarpEpi0) {
        // ------------------------------------------------------------ softmax
        warpgroup_reg_alloc<C::REG_SOFT>();
        const int sw = warp;                     // softmax warp 0..3 = its tensor-memory lane quarter
        const int row = sw * 32 + lane;          // this thread's lane: a token of S^T, a dim of O^T
        const uint32_t taddr = tmem + ((uint32_t)(sw * 32) << 16);
        const uint32_t col_o = C::COL_O;
        uint32_t gt = 0, un = 0;
        // Descriptor of unit `it` (the same in all four warps); false when a wait gave up.
        auto fetch = [&](uint32_t it, UnitDesc& u) {
            const uint32_t qs = it % C::NQ;
            const bool ok = mbar_wait_warp(&sm.u_full[qs], (it / C::NQ) & 1);
            u.seq = -1;
            if (ok) {
                u = sm.unit[qs];
                __syncwarp();
                if (lane == 0) mbar_arrive(&sm.u_empty[qs]);
            }
            return !consumers_any(!ok, kSoftThreads);
        };
        UnitDesc u;
        bool failed = !fetch(0, u);
        // un: units handed to the epilogue warps so far (the current unit's index)
        while (!failed && u.seq >= 0) {
            // mref[n]: the reference of row n's weights, p = 2^(y - mref) for the score y in
            // log2 units.  When it moves it is set kSlack above the largest score seen, and
            // it moves only when a score passes it, so weights stay <= 1 and O^T rarely
            // needs rescaling; the result does not depend on the reference.  -inf: the row
            // has seen no token yet.  ls: this thread's share of the row's weight sum.
            float mref[RPAD], ls[RPAD];
#pragma unroll
            for (int n = 0; n < RPAD; ++n) {
                mref[n] = -INFINITY;
                ls[n] = 0.f;
            }
            const int32_t ntiles = (u.tok1 - u.tok0 + kTok - 1) / kTok;
            bool bad = false;   // a wait of this warp gave up
            for (int32_t j = 0; j < ntiles; ++j, ++gt) {
                const uint32_t b = gt & 1;
                const int32_t tile0 = u.tok0 + j * kTok;
                const int32_t tok = tile0 + row;
                const bool ok = !bad && mbar_wait_warp(&sm.s_full[b], (gt >> 1) & 1);
                // causal limit: query token jq sees tokens below len - q_len + jq + 1, so this
                // thread's token is seen from query token jmin on, i.e. by the unit's rows
                // n >= jmin * group - row0 (row n is query token (row0 + n) / group); and
                // never past the unit's last token
                const int32_t jmin = max(tok - (u.len - p.q_len), 0);
                const int32_t nmin = tok < u.tok1 ? jmin * p.group - u.row0 : RPAD;
                // the tile's scores (S^T column of this thread's token), in log2 units and
                // masked; S^T stays in tensor memory until this tile's P^T is published
                auto scores = [&](float (&y)[RPAD]) {
#pragma unroll
                    for (int h = 0; h < RPAD / 16; ++h) {
                        float s16[16];
                        tmem_ld16(taddr + C::COL_S + b * RPAD + 16 * h, s16);
                        tmem_wait_ld();
#pragma unroll
                        for (int i = 0; i < 16; ++i) y[16 * h + i] = s16[i];
                    }
#pragma unroll
                    for (int n = 0; n < RPAD; ++n) y[n] = n >= nmin ? y[n] * p.scale_log2 : -INFINITY;
                };
                // x[n]: exponent of the token's weight in row n, y - mref; a positive one
                // means the reference must move
                float x[RPAD];
                bool need = false;
                if (ok) {
                    tmem_fence_after_sync();
#pragma unroll
                    for (int h = 0; h < RPAD / 16; ++h) {
                        float s16[16];
                        tmem_ld16(taddr + C::COL_S + b * RPAD + 16 * h, s16);
                        tmem_wait_ld();
#pragma unroll
                        for (int i = 0; i < 16; ++i) x[16 * h + i] = s16[i];
                    }
                    float xmax = -INFINITY;
                    if (nmin <= 0) {   // every row sees the token
#pragma unroll
                        for (int n = 0; n < RPAD; ++n) {
                            x[n] = fmaf(x[n], p.scale_log2, -mref[n]);
                            xmax = fmaxf(xmax, x[n]);
                        }
                    } else {
#pragma unroll
                        for (int n = 0; n < RPAD; ++n) {
                            x[n] = n >= nmin ? fmaf(x[n], p.scale_log2, -mref[n]) : -INFINITY;
                            xmax = fmaxf(xmax, x[n]);
                        }
                    }
                    need = xmax > 0.f;
                }
                // one barrier per tile: abort together, or move the references together
                if (consumers_any(!ok || need, kSoftThreads)) {
                    if (consumers_any(!ok, kSoftThreads)) {
                        failed = true;
                        break;
                    }
                    scores(x);
                    float cmax[RPAD];
#pragma unroll
                    for (int n = 0; n < RPAD; ++n) cmax[n] = x[n];
                    const float wmax = warp_transpose_reduce<RPAD, true>(cmax, lane);
                    if (lane < RPAD) sm.red[b][lane][sw] = wmax;
                    named_bar_sync(kBarSoft, kSoftThreads);
                    bool rescale = false;
                    float alpha[RPAD];
#pragma unroll
                    for (int n = 0; n < RPAD; ++n) {
                        const float4 r4 = *reinterpret_cast<const float4*>(sm.red[b][n]);
                        const float tmax = fmaxf(fmaxf(r4.x, r4.y), fmaxf(r4.z, r4.w));
                        const float mn = tmax > mref[n] ? tmax + kSlack : mref[n];
                        alpha[n] = mref[n] == -INFINITY ? 0.f : fast_exp2(mref[n] - mn);
                        rescale |= (j > 0 && mref[n] != -INFINITY && mn != mref[n]);
                        ls[n] *= alpha[n];
                        mref[n] = mn;
                        x[n] = mn == -INFINITY ? -INFINITY : x[n] - mn;
                    }
                    if (rescale) {
                        // O^T row (head dim `row`) times alpha per query-row column, once the
                        // PV of the previous tile has landed
                        const bool okr = mbar_wait_warp(&sm.pv_done[(gt - 1) & 1], ((gt - 1) >> 1) & 1);
                        if (okr) {
                            tmem_fence_after_sync();
                            // (column c of O^T is row c % RPAD: O_hi, then O_lo)
#pragma unroll
                            for (int h = 0; h < C::NPV / 16; ++h) {
                                float o16[16];
                                const uint32_t ob = taddr + col_o + (un & 1) * C::NPV + 16 * h;
                                tmem_ld16(ob, o16);
                                tmem_wait_ld();
#pragma unroll
                                for (int i = 0; i < 16; ++i) o16[i] *= alpha[(16 * h + i) % RPAD];
                                tmem_st16(ob, o16);
                            }
                            tmem_wait_st();
                        }
                        bad |= !okr;
                    }
                    named_bar_sync(kBarSoft, kSoftThreads);   // red[b] is read by all
                }
#pragma unroll
                for (int n = 0; n < RPAD; ++n) {
                    x[n] = fast_exp2(x[n]);   // masked, or no token seen by the row yet: 0
                    ls[n] += x[n];
                }
                // P^T buffer gt % NP was last read by the PV of tile gt - NP
                uint8_t* const pbuf = sm.p[gt % C::NP];
                if (!bad && gt >= (uint32_t)C::NP) {
                    const uint32_t t = gt - C::NP;
                    bad = !mbar_wait_warp(&sm.pv_done[t & 1], (t >> 1) & 1);
                }
                // the last tile of a unit may stop inside a block: zero the V rows past the
                // unit (they may hold anything, NaN included; 0 x NaN must not reach O)
                const int32_t valid = u.tok1 - tile0;
                if (!bad && valid < kTok) {
                    const uint32_t vs = gt % C::NV;
                    bad = !mbar_wait_warp(&sm.v_full[vs], (gt / C::NV) & 1);
                    if (!bad && row >= valid) {
                        // chunk order rotated by row: neighbouring lanes hit different banks
#pragma unroll
                        for (int h = 0; h < 2; ++h)
#pragma unroll
                            for (int c = 0; c < 8; ++c)
                                *reinterpret_cast<uint4*>(sm.v[vs] + h * kHalf + row * 128 +
                                                          (((c + row) & 7) << 4)) = make_uint4(0u, 0u, 0u, 0u);
                    }
                }
                if (bad) continue;   // the next barrier makes the abort uniform
                // P^T row of this thread's token: the weights rounded to the 16-bit type in
                // pairs, and for bf16 the rounding remainders as a second term
                {
                    uint32_t w2[C::NPV / 2];
#pragma unroll
                    for (int i = 0; i < RPAD / 2; ++i) w2[i] = pack2<C::kBf16>(x[2 * i], x[2 * i + 1]);
                    if constexpr (C::PSPLIT == 2) {
#pragma unroll
                        for (int i = 0; i < RPAD / 2; ++i) {
                            float h0, h1;
                            unpack2<true>(w2[i], h0, h1);
                            w2[RPAD / 2 + i] = pack2<true>(x[2 * i] - h0, x[2 * i + 1] - h1);
                        }
                    }
                    constexpr int kChunks = C::PROW / 16;
                    const int swz = (row * (int)C::PROW >> 7) & (kChunks - 1);
                    uint8_t* const prow = pbuf + row * C::PROW;
#pragma unroll
                    for (int c = 0; c < kChunks; ++c)
                        *reinterpret_cast<uint4*>(prow + ((c ^ swz) << 4)) =
                            make_uint4(w2[4 * c], w2[4 * c + 1], w2[4 * c + 2], w2[4 * c + 3]);
                }
                fence_proxy_async_smem();   // P^T and zeroed V rows -> the tensor core
                tmem_fence_before_sync();
                __syncwarp();
                if (lane == 0) mbar_arrive(&sm.p_full[b]);
            }
            if (!failed && consumers_any(bad, kSoftThreads)) failed = true;
            if (failed) break;
            // ---- hand the unit to the epilogue warps: descriptor, row references and this
            // warp's column exp-sums into slot un & 1, once they have read that slot's
            // previous unit (and its O^T buffer); O^T stays in tensor memory
            const uint32_t es = un & 1;
            bool ok = mbar_wait_warp(&sm.o_empty[es], ((un >> 1) & 1) ^ 1);
            if (ok) {
                float lsum[RPAD];
#pragma unroll
                for (int n = 0; n < RPAD; ++n) lsum[n] = ls[n];
                const float wsum = warp_transpose_reduce<RPAD, false>(lsum, lane);
                if (lane < RPAD) sm.lred[es][lane][sw] = wsum;
                if (sw == 0) {
                    float mr = 0.f;
#pragma unroll
                    for (int n = 0; n < RPAD; ++n) mr = n == lane ? mref[n] : mr;
                    if (lane < RPAD) sm.mrow[es][lane] = mr;
                    if (lane == 0) sm.eunit[es] = u;
                }
                __syncwarp();
                if (lane == 0) mbar_arrive(&sm.e_full[es]);
            }
            if (consumers_any(!ok, kSoftThreads)) {
                failed = true;
                break;
            }
            ++un;
            UnitDesc nu;
            if (!fetch(un, nu)) {
                failed = true;
                break;
            }
            u = nu;
        }
        // the epilogue warps stop at a slot without a sequence (the slot after the last
        // unit handed over)
        {
            const uint32_t es = un & 1;
            const bool ok = mbar_wait_warp(&sm.o_empty[es], ((un >> 1) & 1) ^ 1);
            if (ok && sw == 0 && lane == 0) sm.eunit[es].seq = -1;
            __syncwarp();
            if (ok && lane == 0) mbar_arrive(&sm.e_full[es]);
        }
        if (failed && lane == 0) {
            flag_error(p.status, PA_DEVERR_TIMEOUT_);
            sm.abort = 1;
        }
    } else {
        // ------------------------------------------------------------ epilogue
        warpgroup_reg_release<C::REG_EPI>();
        const int ew = warp - kWarpEpi0;         // epilogue warp 0..3 = its tensor-memory lane quarter
        const int row = ew * 32 + lane;          // this thread's head dim of O^T
        const int tid = ew * 32 + lane;
        const uint32_t taddr = tmem + ((uint32_t)(ew * 32) << 16);
        bool failed = false;
        for (uint32_t un = 0;; ++un) {
            const uint32_t es = un & 1, eph = (un >> 1) & 1;
            // the unit, its row references and exp-sums (row n's in lane n < RPAD)
            bool ok = mbar_wait_warp(&sm.e_full[es], eph);
            UnitDesc u;
            u.seq = -1;
            float L_row = 0.f, m_row = 0.f;
            if (ok) {
                u = sm.eunit[es];
                if (lane < RPAD) {
                    const float4 l4 = *reinterpret_cast<const float4*>(sm.lred[es][lane]);
                    L_row = (l4.x + l4.y) + (l4.z + l4.w);
                    m_row = sm.mrow[es][lane];
                }
            }
            if (consumers_any(!ok, kEpiThreads, kBarEpi)) {
                failed = true;
                break;
            }
            if (u.seq < 0) break;
            const int32_t ntiles = (u.tok1 - u.tok0 + kTok - 1) / kTok;
            // O^T column n (and column RPAD + n, the second term for bf16) is query row
            // u.row0 + n; this thread holds head dim `row`.  Rows go out 16 at a time.  A
            // unit without tiles issued no PV: its rows are 0.
            ok = mbar_wait_warp(&sm.o_full[es], eph);
            if (consumers_any(!ok, kEpiThreads, kBarEpi)) {
                failed = true;
                break;
            }
            tmem_fence_after_sync();
            const bool final_out = u.pslot < 0;
            const float inv_row = L_row > 0.f ? p.out_scale / L_row : 0.f;   // row `lane`'s
            const size_t pr0 = final_out ? 0 : part_row(p, u, u.pslot, 0);
#pragma unroll
            for (int g = 0; g < RPAD / 16; ++g) {
                float o[16];
                tmem_ld16(taddr + C::COL_O + es * C::NPV + 16 * g, o);
                tmem_wait_ld();
                if constexpr (C::PSPLIT == 2) {
                    float lo[16];
                    tmem_ld16(taddr + C::COL_O + es * C::NPV + RPAD + 16 * g, lo);
                    tmem_wait_ld();
#pragma unroll
                    for (int i = 0; i < 16; ++i) o[i] += lo[i];
                }
#pragma unroll
                for (int i = 0; i < 16; ++i) o[i] = ntiles > 0 ? o[i] : 0.f;
                if (g == RPAD / 16 - 1) {
                    tmem_fence_before_sync();
                    __syncwarp();
                    if (lane == 0) mbar_arrive(&sm.o_empty[es]);   // O^T buffer and slot es are free
                }
                if (final_out) {
                    // normalised and rounded, staged [row][dim], then written out in 16-byte
                    // pieces (an output row is 256 contiguous bytes)
#pragma unroll
                    for (int i = 0; i < 16; ++i)
                        sm.ostage[i][row] = to16<C::kBf16>(o[i] * __shfl_sync(0xffffffffu, inv_row, 16 * g + i));
                    named_bar_sync(kBarEpi, kEpiThreads);
                    constexpr int kPieces = 16 * kD * 2 / 16;
#pragma unroll
                    for (int k = 0; k < kPieces / kEpiThreads; ++k) {
                        const int c = tid + kEpiThreads * k, i = c >> 4, piece = c & 15;
                        if (16 * g + i < u.nrows) {
                            uint16_t* dst = reinterpret_cast<uint16_t*>(p.out) +
                                            mq_out_row(p, u.seq, u.kvh, u.row0 + 16 * g + i) * kD + piece * 8;
                            *reinterpret_cast<uint4*>(dst) =
                                *reinterpret_cast<const uint4*>(&sm.ostage[i][piece * 8]);
                        }
                    }
                    named_bar_sync(kBarEpi, kEpiThreads);   // ostage is reused
                } else {
                    // unnormalised partial rows of this partition
#pragma unroll
                    for (int i = 0; i < 16; ++i)
                        if (16 * g + i < u.nrows) p.part_acc[(pr0 + 16 * g + i) * kD + row] = o[i];
                }
            }
            if (!final_out) {
                // (m, l) of each row
                if (ew == 0 && lane < u.nrows) p.part_ml[pr0 + lane] = make_float2(m_row, L_row);
                // count this partition; the last of the (sequence, kv head, row chunk)
                // merges all partials by log-sum-exp
                __threadfence();
                named_bar_sync(kBarEpi, kEpiThreads);
                if (tid == 0) {
                    const size_t pair = ((size_t)u.seq * Hkv + u.kvh) * (size_t)RC + u.row0 / RPAD;
                    sm.last_flag = atomicAdd(&p.arrive[pair], 1) == u.nparts - 1;
                }
                named_bar_sync(kBarEpi, kEpiThreads);
                if (sm.last_flag) {
                    __threadfence();
                    for (int n = 0; n < u.nrows; ++n) {
                        float M = -INFINITY, den = 0.f, acc = 0.f;
                        for (int q = 0; q < u.nparts; ++q) {
                            const size_t pr = part_row(p, u, u.pbase + q, n);
                            const float2 ml = __ldcg(&p.part_ml[pr]);
                            const float a = __ldcg(&p.part_acc[pr * kD + row]);
                            const float Mn = fmaxf(M, ml.x);
                            const float f = state_weight(M, Mn), wq = state_weight(ml.x, Mn);
                            den = den * f + wq * ml.y;
                            acc = acc * f + wq * a;
                            M = Mn;
                        }
                        const float inv = den > 0.f ? p.out_scale / den : 0.f;
                        reinterpret_cast<uint16_t*>(p.out)[mq_out_row(p, u.seq, u.kvh, u.row0 + n) * kD + row] =
                            to16<C::kBf16>(acc * inv);
                    }
                }
            }
            named_bar_sync(kBarEpi, kEpiThreads);   // last_flag is reused
        }
        if (failed && lane == 0) {
            flag_error(p.status, PA_DEVERR_TIMEOUT_);
            sm.abort = 1;
        }
    }

    // Teardown.  After an abort, copies may still be landing in shared memory: wait
    // (bounded) for every stage whose TMA was issued but never fed to an MMA.
    __syncthreads();
    if (threadIdx.x == 0 && sm.abort) {
        for (int i = 0; i < C::NK; ++i)
            if (sm.k_issued[i] > sm.k_done[i]) (void)mbar_wait(&sm.k_full[i], sm.k_done[i] & 1);
        for (int i = 0; i < C::NV; ++i)
            if (sm.v_issued[i] > sm.v_done[i]) (void)mbar_wait(&sm.v_full[i], sm.v_done[i] & 1);
    }
    __syncthreads();
    if (warp == kWarpMma) {
        tmem_fence_after_sync();
        tmem_dealloc(tmem, C::TMEM_COLS);
    }
}

}  // namespace tc
}  // namespace pa
