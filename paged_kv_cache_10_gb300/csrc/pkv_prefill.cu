// pkv_prefill.cu -- paged (chunked) prefill attention on the 5th-generation
// tensor cores (tcgen05, accumulators in tensor memory).
//
// Prefill processes a prompt's tokens at once; chunked prefill cuts a long
// prompt into chunks of at most a token budget that run in successive
// iterations ("vLLM 高性能大语言模型推理引擎深度技术评估与分布式架构展望",
// "PagedAttention 内存管理与核心数据结构" and its scheduling section on chunked
// prefill).  A chunk's query tokens attend causally to the sequence's whole
// history in the paged pool -- earlier chunks and their own chunk up to
// themselves -- gathered through the block table like decode.
//
// A unit of work is two Q tiles of 128 query rows of one (sequence, KV
// head), each 128 / G tokens x the G query heads of the group, so every
// key / value tile feeds all heads that read it and both Q tiles.  Per
// 128-key tile (8 pool blocks):
//   S = Q K^T    tcgen05.mma, M = 128 rows, N = 128 keys, fp32 in tensor memory
//   P = exp2(S * scale * log2 e - m)    one thread per row, from tensor memory
//   O += P V     tcgen05.mma with P from tensor memory, O in tensor memory;
//                P as a 16-bit head plus a 16-bit tail (two MMAs into O), so
//                the probabilities keep 16 (bf16) or 22 (f16) significant bits
// Warp roles: warp 3 claims units and loads their Q tiles (3-D TMA map);
// warp 0 streams the key tiles through a 3-stage ring and warp 2 the value
// tiles through a 2-stage ring (per pool block, by the pool's 2-D map);
// warp 1 issues the MMAs and owns the tensor memory; warps 4-7 and 8-11 run
// the online softmax, the O corrections and the epilogue of Q tiles A and
// B, one thread per query row, with packed two-lane fp32 arithmetic.
// P_j (head and tail) is written back over S_j, where the P V MMAs read it as their A
// operand; the two Q tiles ping-pong, so one tile's MMAs run while the
// other's softmax works.  The running max is rebased only when it grows by
// more than 2^8, which keeps every probability <= 256 and skips most O
// corrections; the final O / l is the same softmax.
#include <algorithm>
#include <atomic>
#include <cstdint>
#include <mutex>
#include <type_traits>

#include "pkv_decode_mma.cuh"  // ex2, pack2, swz128, fence_proxy_async_smem
#include "pkv_tcgen05.cuh"

namespace pkv {
namespace {

constexpr int kTileM = 128;     // query rows per Q tile (two Q tiles per CTA)
constexpr int kTileN = 128;     // keys per tile
constexpr int kKStages = 3;     // key ring depth
constexpr int kVStages = 2;     // value ring depth
constexpr int kColBlock = kTileM * 128;  // one 64-column block of a 128-row 16-bit operand (16 KB)
constexpr int kBlockTileBytes = kBlockSize * 128;  // 16 rows x 128 bytes
// Three warpgroups: warps 0-3 load (0: Q and keys, 2: values), issue the
// MMAs (1) or idle (3); warps 4-7 run the softmax of Q tile A, warps 8-11 of
// Q tile B.  setmaxnreg moves registers from the first to the other two:
// 128 x 104 + 256 x 192 <= 384 x 168, the launch's allocation.
constexpr int kThreads = 384;
constexpr int kLoadRegs = 104;
constexpr int kSoftmaxRegs = 192;
static_assert(128 * kLoadRegs + 256 * kSoftmaxRegs <= kThreads * (65536 / kThreads / 8 * 8), "register split");
constexpr int kSoftmaxWarps = 4;  // per Q tile
constexpr float kRebase = 8.0f;   // log2 units

// Persistent prefill: each CTA claims units from a counter and publishes
// them to its warps through a ring of kUnitSlots slots; 11 warps read each
// slot (the K, V and MMA warps and the 8 softmax warps).
constexpr int kUnitSlots = 4;
constexpr int kUnitReaders = 11;

// q_full, q_empty, k_full[3], k_empty[3], v_full[2], v_empty[2], v_zero[2], s_full[2 tiles],
// p_full[2 tiles], o_done[2 tiles], drain, u_full[4], u_empty[4]
constexpr int kNumBars = 2 + 2 * kKStages + 3 * kVStages + 2 + 2 + 2 + 1 + 2 * kUnitSlots;

// Shared-memory layout for head_size D (64 or 128): operands are 128 rows x
// D 16-bit elements in D / 64 column blocks of 128-byte rows.
template <int D>
struct Tile {
    static_assert(D == 64 || D == 128, "head_size");
    static constexpr int kDB = D / 64;          // 64-column blocks per row
    static constexpr int kOp = kTileM * D * 2;  // one 128 x D operand
    static constexpr int kOffQ = 0;             // Q tiles A, B
    static constexpr int kOffK = kOffQ + 2 * kOp;
    static constexpr int kOffV = kOffK + kKStages * kOp;
    static constexpr int kOffBar = kOffV + kVStages * kOp;
    static constexpr int kOffMisc = kOffBar + kNumBars * 8;
    static constexpr int kUnitBytes = 48;  // one published unit (sizeof(Unit) rounded up)
    static constexpr int kSmemBytes = kOffMisc + 8 + kUnitSlots * kUnitBytes + 1024;  // tmem slot, abort flag,
                                                                                       // unit ring; alignment slack
    static_assert(kSmemBytes <= 227 * 1024, "shared memory");
};

struct PrefillParams {
    const int32_t* query_start;  // [S + 1]
    const int32_t* block_tables; // [S][MB]
    const int32_t* seq_lens;     // [S], counting the new tokens
    void* out;                   // [T][Hq][D]
    int32_t S, T, Hq, Hkv, MB, NB;
    int32_t G, TT;               // heads per KV head, tokens per CTA (128 / G)
    int32_t num_qtiles;          // CTAs per (sequence, KV head) along the queries
    int32_t max_query_len;       // the caller's bound on every chunk
    const int32_t* work;         // [num_work] units s * num_qtiles + qt in start order, or null
    int32_t num_work;
    float qk_scale;              // scale * log2(e) (* k_scale for a staged fp8 pool)
    float o_scale = 1.f;         // factor on O / l: v_scale for a staged fp8 pool
    int32_t out_v8 = 0;          // out is 32-byte aligned: 32-byte stores in the epilogue
    unsigned int* err;
    // cascade prefix pass only
    const int32_t* group_offsets;  // [groups + 1]
    const int32_t* group_members;  // batch rows
    const int32_t* group_blocks;   // shared leading blocks per group
    float* part_m;                 // partials [S][Hq][NP] (log2 units), [S][Hq][NP], [S][Hq][NP][D]
    float* part_l;
    float* part_o;
    int32_t NP, row_chunks;
    // prefill: the launch's scheduling counters (g_prefill_sched slot)
    int32_t sched_slot;
};

// Unit-claim counters of the persistent prefill, one pair (next unit, CTAs
// finished) per launch slot.  Zero at load; the last CTA of a launch puts its
// pair back to zero, so a launch (or a graph replay) always starts from 0.
// The host hands out slots round-robin: launches that run at the same time
// take different slots unless kSchedSlots of them overlap.
constexpr int kSchedSlots = 1024;
__device__ unsigned int g_prefill_sched[2 * kSchedSlots];

__device__ __forceinline__ bool warp_all(bool v) { return __all_sync(0xffffffffu, v); }

// One 32-byte store (p 32-byte aligned): a whole L2 sector per thread.
__device__ __forceinline__ void st_global_v8(void* p, const uint32_t (&w)[8]) {
    asm volatile("st.global.v8.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8};" ::"l"(p), "r"(w[0]), "r"(w[1]),
                 "r"(w[2]), "r"(w[3]), "r"(w[4]), "r"(w[5]), "r"(w[6]), "r"(w[7])
                 : "memory");
}

// Two-lane fp32 arithmetic (one instruction, each lane rounded as the scalar
// operation) and a three-input maximum.
__device__ __forceinline__ float2 ffma2(float2 a, float2 b, float2 c) {
    float2 d;
    asm("{\n\t.reg .b64 ra, rb, rc, rd;\n\t"
        "mov.b64 ra, {%2, %3};\n\tmov.b64 rb, {%4, %5};\n\tmov.b64 rc, {%6, %7};\n\t"
        "fma.rn.f32x2 rd, ra, rb, rc;\n\tmov.b64 {%0, %1}, rd;\n\t}"
        : "=f"(d.x), "=f"(d.y)
        : "f"(a.x), "f"(a.y), "f"(b.x), "f"(b.y), "f"(c.x), "f"(c.y));
    return d;
}

__device__ __forceinline__ float2 fadd2(float2 a, float2 b) {
    float2 d;
    asm("{\n\t.reg .b64 ra, rb, rd;\n\t"
        "mov.b64 ra, {%2, %3};\n\tmov.b64 rb, {%4, %5};\n\t"
        "add.rn.f32x2 rd, ra, rb;\n\tmov.b64 {%0, %1}, rd;\n\t}"
        : "=f"(d.x), "=f"(d.y)
        : "f"(a.x), "f"(a.y), "f"(b.x), "f"(b.y));
    return d;
}

__device__ __forceinline__ float2 fmul2(float2 a, float2 b) {
    float2 d;
    asm("{\n\t.reg .b64 ra, rb, rd;\n\t"
        "mov.b64 ra, {%2, %3};\n\tmov.b64 rb, {%4, %5};\n\t"
        "mul.rn.f32x2 rd, ra, rb;\n\tmov.b64 {%0, %1}, rd;\n\t}"
        : "=f"(d.x), "=f"(d.y)
        : "f"(a.x), "f"(a.y), "f"(b.x), "f"(b.y));
    return d;
}

// Two probabilities as a 16-bit head pair and a 16-bit tail pair (the
// head's remainder, rounded once): head + tail keeps 16 (bf16) or 22 (f16)
// significant bits.  bf16: the head is the top half of each float32 (a
// truncation: one byte permute), so the remainder x - head is the exact low
// half; f16: the head is rounded to nearest and the remainder taken exactly.
template <bool BF>
__device__ __forceinline__ void split2(float2 a, uint32_t& head, uint32_t& tail) {
    float2 t;
    if constexpr (BF) {
        const uint32_t ux = __float_as_uint(a.x), uy = __float_as_uint(a.y);
        head = __byte_perm(ux, uy, 0x7632);
        t = fadd2(a, make_float2(__uint_as_float((ux & 0xffff0000u) ^ 0x80000000u),
                                 __uint_as_float((uy & 0xffff0000u) ^ 0x80000000u)));
    } else {
        head = pack2<false>(a.x, a.y);
        const float2 r = __half22float2(*reinterpret_cast<const __half2*>(&head));
        t = fadd2(a, make_float2(-r.x, -r.y));
    }
    tail = pack2<BF>(t.x, t.y);
}

__device__ __forceinline__ float fmax3(float a, float b, float c) {
    float d;
    asm("max.f32 %0, %1, %2, %3;" : "=f"(d) : "f"(a), "f"(b), "f"(c));
    return d;
}

// D[tmem] (+)= A[tmem] * B[smem]: the A operand (M = 128 lanes) read from
// tensor memory, two 16-bit elements per 32-bit column (column c of lane r
// holds A[r][2c] in its low half, A[r][2c + 1] in its high half), so one
// K = 16 step spans 8 columns.
__device__ __forceinline__ void mma_f16_tmem_a(uint32_t d_tmem, uint32_t a_tmem, uint64_t bdesc, uint32_t idesc,
                                               bool accumulate) {
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "setp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n\t}" ::"r"(d_tmem),
        "r"(a_tmem), "l"(bdesc), "r"(idesc), "r"(accumulate ? 1u : 0u)
        : "memory");
}

__device__ __forceinline__ void setmaxnreg_dec() {
    asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;" ::"n"(kLoadRegs));
}
__device__ __forceinline__ void setmaxnreg_inc() {
    asm volatile("setmaxnreg.inc.sync.aligned.u32 %0;" ::"n"(kSoftmaxRegs));
}

// One unit of work: the rows of a Q tile pair and the keys they need.
struct Unit {
    const int32_t* bt;  // block table, from the unit's first key block
    int kv_end[2];      // keys Q tile X needs (0: the tile has no rows)
    int h;              // KV head
    int q0, n, ctx, t0;  // prefill: the sequence's first row in q / out, its new tokens, the
                         // tokens before them, the first token of Q tile A
};

// Prefill unit number lin: unit work[lin / Hkv] of the host plan (or of the
// default order: each (sequence, KV head) from its last query tiles down)
// for KV head lin % Hkv.  False when the unit has no rows or its sequence's
// bounds are inconsistent (reported when rep).
__device__ bool prefill_unit(const PrefillParams& p, int64_t lin, int RQ, bool rep, Unit& u) {
    int s, qt;
    if (p.work) {
        const int w = __ldg(p.work + lin / p.Hkv);
        u.h = static_cast<int>(lin % p.Hkv);
        if (w < 0 || w >= p.S * p.num_qtiles) {
            if (rep) report(p.err, PKV_DEVERR_SEQ_LEN);
            return false;
        }
        s = w / p.num_qtiles;
        qt = w % p.num_qtiles;
    } else {
        qt = p.num_qtiles - 1 - static_cast<int>(lin % p.num_qtiles);
        u.h = static_cast<int>((lin / p.num_qtiles) % p.Hkv);
        s = static_cast<int>(lin / (static_cast<int64_t>(p.num_qtiles) * p.Hkv));
    }
    u.q0 = __ldg(p.query_start + s);
    const int q1 = __ldg(p.query_start + s + 1);
    u.n = q1 - u.q0;
    const int L = __ldg(p.seq_lens + s);
    if (u.q0 < 0 || u.n < 0 || q1 > p.T || L < u.n || L > p.MB * kBlockSize) {
        if (rep) report(p.err, PKV_DEVERR_SEQ_LEN);
        return false;
    }
    if (u.n > p.max_query_len && rep) report(p.err, PKV_DEVERR_SEQ_LEN);
    u.t0 = qt * 2 * RQ;
    if (u.t0 >= u.n) return false;
    u.ctx = L - u.n;  // tokens before this chunk
    for (int X = 0; X < 2; ++X) {
        const int tx = u.t0 + X * RQ;
        u.kv_end[X] = tx < u.n ? u.ctx + tx + min(RQ, u.n - tx) : 0;
    }
    u.bt = p.block_tables + static_cast<int64_t>(s) * p.MB;
    return true;
}

// Waits for unit k in the ring slot k % kUnitSlots, copies it and hands the
// slot back; false on timeout.  A unit with h < 0 ends the list.  Called by
// one thread (warp 1) or by a whole warp (every lane waits; lane 0 hands
// back).
__device__ __forceinline__ bool take_unit(uint64_t* u_full, uint64_t* u_empty, const Unit* ring, int k,
                                          bool whole_warp, Unit& u) {
    const int slot = k % kUnitSlots;
    bool ok = mbar_wait(u_full + slot, (k / kUnitSlots) & 1);
    if (whole_warp) ok = __all_sync(0xffffffffu, ok);
    if (!ok) return false;
    u = ring[slot];
    if (whole_warp) __syncwarp();
    if (!whole_warp || (threadIdx.x & 31) == 0) tc::arrive(u_empty + slot);
    return true;
}

// kPrefix = false: causal prefill, persistent.  The grid has one CTA per SM
// (or per unit, when there are fewer); each CTA claims units in list order
// from a counter, so the longest units of the host plan start first and an
// SM that finishes early takes the next one.  Warp 3 claims unit k + 1 and
// loads its Q tiles while the other warps still work on unit k, and the K / V
// rings run across unit boundaries, so the next unit's loads overlap this
// unit's last tiles and epilogue.  Q tile X (X = 0, 1) holds 128 / G tokens x
// the G heads of one (sequence, KV head), tokens [t0 + X * TT, ...); keys 0 ..
// each row's position; normalised output.
// kPrefix = true: the cascade decode's shared-prefix pass, one unit per CTA;
// Q tile X holds 128 / G members x G heads of one (group, KV head); keys =
// one partition of the group's shared blocks (no causal mask); split-K
// partials.
template <typename T, int D, bool kPrefix>
__global__ void __launch_bounds__(kThreads, 1)
    prefill_tc_kernel(const PrefillParams p, const __grid_constant__ CUtensorMap tmq,
                      const __grid_constant__ CUtensorMap tmk, const __grid_constant__ CUtensorMap tmv) {
    constexpr bool kBF = std::is_same<T, BF16>::value;
    // cascade decode: the own-token decode after this grid reads nothing it
    // writes and may start at once
    if constexpr (kPrefix) allow_dependent_launch();
    using TL = Tile<D>;
    constexpr int kOffQ = TL::kOffQ, kOffK = TL::kOffK, kOffV = TL::kOffV, kOffMisc = TL::kOffMisc;
    constexpr int kOpBytes = TL::kOp, kDB = TL::kDB;
    extern __shared__ unsigned char smem_raw[];
    unsigned char* sm = smem_raw + ((1024 - (smem_addr(smem_raw) & 1023)) & 1023);
    uint64_t* q_full = reinterpret_cast<uint64_t*>(sm + TL::kOffBar);
    uint64_t* q_empty = q_full + 1;
    uint64_t* k_full = q_empty + 1;          // [kKStages]
    uint64_t* k_empty = k_full + kKStages;   // [kKStages]
    uint64_t* v_full = k_empty + kKStages;   // [kVStages]
    uint64_t* v_empty = v_full + kVStages;   // [kVStages]
    uint64_t* v_zero = v_empty + kVStages;   // [kVStages]
    uint64_t* s_full = v_zero + kVStages;    // [Q tile]
    uint64_t* p_full = s_full + 2;           // [Q tile]
    uint64_t* o_done = p_full + 2;           // [Q tile]
    uint64_t* drain = o_done + 2;
    uint64_t* u_full = drain + 1;            // [kUnitSlots]
    uint64_t* u_empty = u_full + kUnitSlots; // [kUnitSlots]
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(sm + kOffMisc);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(sm + kOffMisc + 4);
    Unit* unit_ring = reinterpret_cast<Unit*>(sm + kOffMisc + 8);  // [kUnitSlots]

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int G = p.G;
    const int RQ = kTileM / G;  // tokens (prefill) or members (prefix) per Q tile
    // prefix pass: this CTA's one unit, fixed by its grid position
    Unit pre{};
    int m0 = 0, members = 0, mrow0 = 0, seq0 = 0, pp = 0;
    if constexpr (kPrefix) {
        pp = blockIdx.x;
        pre.h = blockIdx.y;
        const int h = pre.h;
        const int grp = blockIdx.z / p.row_chunks, chunk = blockIdx.z % p.row_chunks;
        m0 = __ldg(p.group_offsets + grp);
        members = __ldg(p.group_offsets + grp + 1) - m0;
        // One Q tile per CTA: the prefix pass is short (a few key tiles per
        // CTA), so more CTAs beat the second tile's overlap.
        mrow0 = chunk * RQ;  // first member of this CTA
        if (mrow0 >= members) return;
        int nb = __ldg(p.group_blocks + grp);
        if (nb < 0 || nb > p.MB) {
            if (threadIdx.x == 0 && pp == 0 && h == 0 && chunk == 0) report(p.err, PKV_DEVERR_SEQ_LEN);
            nb = nb < 0 ? 0 : p.MB;
        }
        seq0 = __ldg(p.group_members + m0);
        const bool bad = seq0 < 0 || seq0 >= p.S;
        if (bad && threadIdx.x == 0 && pp == 0 && h == 0 && chunk == 0) report(p.err, PKV_DEVERR_SEQ_LEN);
        const int b0 = pp * kPrefixPartitionBlocks;
        if (b0 >= nb || bad) {
            // this partition lies past the group's prefix (another group's
            // prefix is longer): empty partials, so the merge reads no stale
            // workspace
            for (int r = threadIdx.x; r < kTileM; r += kThreads) {
                const int mi = mrow0 + r / G;
                if (mi >= members) continue;
                const int b = __ldg(p.group_members + m0 + mi);
                if (b < 0 || b >= p.S) continue;
                const int64_t prow = (static_cast<int64_t>(b) * p.Hq + h * G + r % G) * p.NP + pp;
                p.part_m[prow] = -INFINITY;
                p.part_l[prow] = 0.f;
                float4* po = reinterpret_cast<float4*>(p.part_o + prow * D);
                for (int d4 = 0; d4 < D / 4; ++d4) po[d4] = make_float4(0.f, 0.f, 0.f, 0.f);
            }
            return;
        }
        const int keys = (min(nb, b0 + kPrefixPartitionBlocks) - b0) * kBlockSize;
        pre.kv_end[0] = keys;
        pre.kv_end[1] = 0;
        pre.bt = p.block_tables + static_cast<int64_t>(seq0) * p.MB + b0;
    }
    // unit k for a reading role: 1 = a unit, 0 = the list has ended, -1 =
    // timeout.  The prefix pass has its one unit and uses no ring.
    auto next_unit = [&](int k, bool whole_warp, Unit& u) -> int {
        if constexpr (kPrefix) {
            u = pre;
            return k == 0 ? 1 : 0;
        } else {
            if (!take_unit(u_full, u_empty, unit_ring, k, whole_warp, u)) return -1;
            return u.h >= 0 ? 1 : 0;
        }
    };
    unsigned int* sched = g_prefill_sched + 2 * p.sched_slot;
    const int64_t total = kPrefix ? 1
                          : (p.work ? static_cast<int64_t>(p.num_work) * p.Hkv
                                    : static_cast<int64_t>(p.num_qtiles) * p.Hkv * p.S);

    if (threadIdx.x == 0) {
        mbar_init(q_full, 1);
        mbar_init(q_empty, 1);
        for (int i = 0; i < kKStages; ++i) {
            mbar_init(k_full + i, 1);
            mbar_init(k_empty + i, 1);
        }
        for (int i = 0; i < kVStages; ++i) {
            mbar_init(v_full + i, 1);
            mbar_init(v_empty + i, 1);
            mbar_init(v_zero + i, 1);
        }
        for (int i = 0; i < 2; ++i) {
            mbar_init(s_full + i, 1);
            mbar_init(p_full + i, kSoftmaxWarps);  // one arrival per softmax warp
            mbar_init(o_done + i, 1);
        }
        mbar_init(drain, 1);
        for (int i = 0; i < kUnitSlots; ++i) {
            mbar_init(u_full + i, 1);
            mbar_init(u_empty + i, kUnitReaders);
        }
        *abort_flag = 0;
        mbar_init_fence();
    }
    if (warp == 1) {
        tc::tmem_alloc(tmem_slot, 512);
        tc::tmem_relinquish();
    }
    tc::fence_before();
    __syncthreads();
    tc::fence_after();
    const uint32_t tmem = *tmem_slot;
    // Prefill launches as a programmatic dependent of the kernel before it
    // (the fp8 staging pass, or the append): the setup above overlaps that
    // kernel's last CTAs, and nothing here reads global memory before it has
    // completed and its writes are visible.
    if constexpr (!kPrefix) wait_primary_grid();
    // tensor-memory columns: S of Q tile X at X * 128 (its first 64 columns
    // then hold that tile's P, two 16-bit probabilities per column); O of Q
    // tile X at 256 + X * 128
    if (warp < 4) {
      setmaxnreg_dec();
      if (warp == 3) {
        // ------------------------------- unit claims and Q loads (warp 3)
        // Claims the next unit with a row, publishes it to the other warps
        // and loads its Q tiles (the S MMAs of the unit before, which read
        // the Q buffers, are complete by then).  When the list is exhausted
        // it publishes an end marker (a unit with h = -1).  The prefix pass
        // publishes nothing: every warp uses the CTA's one unit.
        const uint64_t pol_q = policy_evict_first();
        int k = 0, qloads = 0;
        bool done = false;
        for (;; ++k) {
            // unit k is claimed once the S MMAs of unit k - 1 are issued (that
            // unit is in its last key tile), so a CTA holds at most one unit
            // ahead and the list stays longest first across the SMs
            if (!kPrefix && k > 0 && !done && !__all_sync(0xffffffffu, mbar_wait(q_empty, (k - 1) & 1))) {
                if (lane == 0) {
                    report(p.err, PKV_DEVERR_TIMEOUT);
                    *abort_flag = 1;
                }
                done = true;  // publishes the end marker
            }
            Unit u{};
            u.h = -1;  // the end of the list unless a claim finds a unit
            if (!done && *abort_flag == 0) {
                if constexpr (kPrefix) {
                    if (k == 0) u = pre;
                } else {
                    bool found = false;
                    for (;;) {
                        unsigned int c = 0;
                        if (lane == 0) c = atomicAdd(sched, 1u);
                        c = __shfl_sync(0xffffffffu, c, 0);
                        if (c >= total) break;
                        if (prefill_unit(p, c, RQ, lane == 0, u)) {
                            found = true;
                            break;
                        }
                    }
                    if (!found) u.h = -1;
                }
            }
            const int slot = k % kUnitSlots;
            if (kPrefix) {
                if (u.h < 0) break;
            } else if (k >= kUnitSlots &&
                       !__all_sync(0xffffffffu, mbar_wait(u_empty + slot, ((k / kUnitSlots) + 1) & 1))) {
                if (lane == 0) {
                    report(p.err, PKV_DEVERR_TIMEOUT);
                    *abort_flag = 1;
                }
                break;
            }
            if (!kPrefix && lane == 0) {
                unit_ring[slot] = u;
                tc::arrive(u_full + slot);
            }
            __syncwarp();
            if (u.h < 0) break;
            const int ntiles = u.kv_end[1] > 0 ? 2 : 1;
            if constexpr (!kPrefix) {
                if (lane == 0) {
                    mbar_arrive_expect_tx(q_full, ntiles * kOpBytes);
                    for (int X = 0; X < ntiles; ++X)
                        for (int dh = 0; dh < kDB; ++dh)
                            tc::tma_load_3d(sm + kOffQ + X * kOpBytes + dh * kColBlock, &tmq, dh * 64, u.h * G,
                                            u.q0 + u.t0 + X * RQ, q_full, pol_q);
                }
            } else {
                // G query rows of each member (its batch row in q); rows of
                // members past the group's end repeat the first member.  All
                // of a lane's member rows are read before any copy is issued.
                constexpr int kMaxPerLane = 2 * kTileM / 32;  // G = 1: 8 members per lane
                int bs[kMaxPerLane];
#pragma unroll
                for (int i = 0; i < kMaxPerLane; ++i) {
                    const int mi = lane + 32 * i;
                    bs[i] = seq0;
                    if (mi < ntiles * RQ && mrow0 + mi < members) bs[i] = __ldg(p.group_members + m0 + mrow0 + mi);
                }
                if (lane == 0) mbar_arrive_expect_tx(q_full, ntiles * kOpBytes);
                __syncwarp();
#pragma unroll
                for (int i = 0; i < kMaxPerLane; ++i) {
                    const int mi = lane + 32 * i;
                    if (mi >= ntiles * RQ) break;
                    int b = bs[i];
                    if (b < 0 || b >= p.S) {
                        report(p.err, PKV_DEVERR_SEQ_LEN);
                        b = seq0;
                    }
                    const int X = mi / RQ, mx = mi - X * RQ;
                    for (int dh = 0; dh < kDB; ++dh)
                        tc::tma_load_3d(sm + kOffQ + X * kOpBytes + dh * kColBlock + mx * G * 128, &tmq, dh * 64,
                                        u.h * G, b, q_full, pol_q);
                }
            }
            ++qloads;
            __syncwarp();
        }
        // the last Q copy has landed before the CTA can exit
        if (qloads > 0 && !mbar_wait(q_full, (qloads - 1) & 1) && lane == 0) report(p.err, PKV_DEVERR_TIMEOUT);
      } else if (warp == 0 || warp == 2) {
        // --------------------------------------------- TMA producers (K, V)
        // Warp 0 streams the key tiles, warp 2 the value tiles, each through
        // its own ring, so a key load never waits for a P V to free a value
        // stage.  Tile g of the CTA (counted across its units) uses stage
        // g % stages.
        const bool is_k = warp == 0;
        const int nst = is_k ? kKStages : kVStages;
        const uint64_t pol_kv = policy_evict_last();  // re-read by other CTAs of the sequence / group
        uint64_t* full = is_k ? k_full : v_full;
        uint64_t* empty = is_k ? k_empty : v_empty;
        const CUtensorMap* map = is_k ? &tmk : &tmv;
        unsigned char* ring = sm + (is_k ? kOffK : kOffV);
        int gt = 0;  // tiles issued by this warp
        bool run = true;
        for (int k = 0; run; ++k) {
            Unit u;
            const int r = next_unit(k, true, u);
            if (r < 0) {
                if (lane == 0) {
                    report(p.err, PKV_DEVERR_TIMEOUT);
                    *abort_flag = 1;
                }
                break;
            }
            if (r == 0) break;
            const int kv_max = max(u.kv_end[0], u.kv_end[1]);
            const int nkt = (kv_max + kTileN - 1) / kTileN;
            const int nblk = (kv_max + kBlockSize - 1) / kBlockSize;
            // block ids 32 at a time (4 tiles), read 4 tiles before their
            // use: lane l holds the id of block 32 * batch + l
            auto load_ids = [&](int batch) {
                const int idx = batch * 32 + lane;
                return idx < nblk ? __ldg(u.bt + idx) : 0;
            };
            int ids_cur = load_ids(0);
            int ids_nxt = load_ids(1);
            for (int j = 0; j < nkt; ++j) {
                const int g = gt;  // this tile's number in the CTA's stream
                const int st = g % nst;
                const int nb_tile = min(8, nblk - j * 8);
                if (j > 0 && (j & 3) == 0) {
                    ids_cur = ids_nxt;
                    ids_nxt = load_ids((j >> 2) + 1);
                }
                int phys = __shfl_sync(0xffffffffu, ids_cur, ((j & 3) << 3) + (lane & 7));
                if (lane < nb_tile && (phys < 0 || phys >= p.NB)) {
                    report(p.err, PKV_DEVERR_BLOCK_ID);
                    phys = 0;
                }
                const int row = (phys * p.Hkv + u.h) * kBlockSize;
                // the stage is free once the MMAs that read it (Q K^T or P V
                // of tile g - nst) have completed
                const bool waited = g < nst || mbar_wait(empty + st, ((g / nst) + 1) & 1);
                if (!warp_all(waited)) {
                    if (lane == 0) {
                        report(p.err, PKV_DEVERR_TIMEOUT);
                        *abort_flag = 1;
                    }
                    run = false;
                    break;
                }
                if (!warp_all(*abort_flag == 0)) {  // uniform across the warp
                    run = false;
                    break;
                }
                if (lane == 0) mbar_arrive_expect_tx(full + st, nb_tile * kDB * kBlockTileBytes);
                __syncwarp();
                if (lane < nb_tile) {
                    unsigned char* d = ring + st * kOpBytes + lane * kBlockTileBytes;
                    for (int dh = 0; dh < kDB; ++dh)
                        tc::tma_load_2d(d + dh * kColBlock, map, dh * 64, row, full + st, pol_kv);
                }
                if (!is_k) {
                    // Value rows at or past the unit's last key get
                    // probability 0, but the pool slots past a sequence's end
                    // (and never-loaded rows) may hold any bits, NaN included,
                    // and 0 * NaN = NaN in the MMA: in the unit's last tile
                    // they are cleared once it has landed.  Every value tile
                    // then completes v_zero of its stage.
                    const int r0 = kv_max - j * kTileN;
                    bool okv = true;
                    if (j == nkt - 1 && r0 < kTileN) {
                        okv = warp_all(mbar_wait(v_full + st, (g / nst) & 1));
                        if (okv) {
                            unsigned char* vb = sm + kOffV + st * kOpBytes;
                            constexpr int kRowChunks = D / 8;  // 16-byte chunks of a row
                            for (int idx = lane; idx < (kTileN - r0) * kRowChunks; idx += 32) {
                                const int r = r0 + idx / kRowChunks, c = idx % kRowChunks;
                                *reinterpret_cast<uint4*>(vb + (c >> 3) * kColBlock + swz128(r, c & 7)) =
                                    make_uint4(0u, 0u, 0u, 0u);
                            }
                            fence_proxy_async_smem();
                        }
                    }
                    __syncwarp();
                    if (lane == 0) {
                        if (!okv) {
                            report(p.err, PKV_DEVERR_TIMEOUT);
                            *abort_flag = 1;
                        }
                        tc::arrive(v_zero + st);
                    }
                }
                gt = g + 1;
            }
        }
        // every copy this warp started has landed before the CTA can exit
        for (int g = gt > nst ? gt - nst : 0; g < gt; ++g)
            if (!mbar_wait(full + g % nst, (g / nst) & 1) && lane == 0)
                report(p.err, PKV_DEVERR_TIMEOUT);
      } else {
        // ------------------------------------------------------- MMA issuer
        // Per unit: S_A(0), S_B(0), then per key tile j: P V_A(j), S_A(j+1),
        // P V_B(j), S_B(j+1).  tcgen05.mma from one thread run in order, so
        // S_X(j+1) overwrites Q tile X's S / P columns only after P V_X(j)
        // has read P_X(j), and the softmax of one Q tile overlaps the MMAs
        // of the other.  The first P V_X of a unit overwrites O_X: it waits
        // for P_X of that unit, which its softmax warps write only after
        // they have read O_X out for the unit before.
        if (lane == 0) {
            const uint32_t idS = tc::idesc_f16(kBF, kTileM, kTileN, false);
            const uint32_t idO = tc::idesc_f16(kBF, kTileM, D, true);
            // Descriptors: bases per Q tile and ring stage, computed once; the
            // k-th 16-element step adds a constant (the start address field
            // is the low 14 bits, >> 4, and every operand sits below 256 KB).
            // Building a descriptor per MMA would make issue, not the tensor
            // core, the limit.
            const uint64_t dQ0 = tc::sdesc_sw128(smem_addr(sm + kOffQ), 16, 1024);
            const uint64_t dQ1 = tc::sdesc_sw128(smem_addr(sm + kOffQ + kOpBytes), 16, 1024);
            const uint64_t dK0 = tc::sdesc_sw128(smem_addr(sm + kOffK), 16, 1024);
            const uint64_t dK1 = tc::sdesc_sw128(smem_addr(sm + kOffK + kOpBytes), 16, 1024);
            const uint64_t dK2 = tc::sdesc_sw128(smem_addr(sm + kOffK + 2 * kOpBytes), 16, 1024);
            const uint64_t dV0 = tc::sdesc_sw128(smem_addr(sm + kOffV), kColBlock, 1024);
            const uint64_t dV1 = tc::sdesc_sw128(smem_addr(sm + kOffV + kOpBytes), kColBlock, 1024);
            bool any_mma = false;
            auto issue_s = [&](int X, int g) {
                any_mma = true;
                const int st = g % kKStages;
                const uint64_t q = X ? dQ1 : dQ0;
                const uint64_t k = st == 0 ? dK0 : (st == 1 ? dK1 : dK2);
                const uint32_t d = tmem + X * kTileN;
#pragma unroll
                for (int kk = 0; kk < D / 16; ++kk) {
                    const uint64_t off = static_cast<uint64_t>(((kk >> 2) * kColBlock + (kk & 3) * 32) >> 4);
                    tc::mma_f16(d, q + off, k + off, idS, kk > 0);
                }
                tc::commit(s_full + X);
            };
            auto issue_pv = [&](int X, int j, int g) {
                const uint64_t v = (g % kVStages) ? dV1 : dV0;
                const uint32_t d = tmem + 256 + X * kTileN, pa = tmem + X * kTileN;
                // P's head (columns 0-63), then its tail (64-127), into the same O
#pragma unroll
                for (int kk = 0; kk < kTileN / 16; ++kk)
                    mma_f16_tmem_a(d, pa + kk * 8, v + static_cast<uint64_t>((kk * kBlockTileBytes) >> 4), idO,
                                   j > 0 || kk > 0);
#pragma unroll
                for (int kk = 0; kk < kTileN / 16; ++kk)
                    mma_f16_tmem_a(d, pa + 64 + kk * 8, v + static_cast<uint64_t>((kk * kBlockTileBytes) >> 4), idO,
                                   true);
                tc::commit(o_done + X);
            };
            bool ok = true;
            int gt = 0;            // key / value tiles of the finished units
            int tp0 = 0, tp1 = 0;  // tiles of Q tiles A and B in the finished units
            for (int k = 0;; ++k) {
                Unit u;
                const int r = next_unit(k, false, u);
                ok = r >= 0;
                if (r <= 0) break;
                const int nt0 = (u.kv_end[0] + kTileN - 1) / kTileN;
                const int nt1 = (u.kv_end[1] + kTileN - 1) / kTileN;
                const int nkt = max(nt0, nt1);
                // this unit's Q tiles and its first keys, then S of both Q tiles
                ok = tc::wait_spin(q_full, k & 1);
                if (ok) ok = tc::wait_spin(k_full + gt % kKStages, (gt / kKStages) & 1);
                if (!ok) break;
                tc::fence_after();
                if (nt0 > 0) issue_s(0, gt);
                if (nt1 > 0) issue_s(1, gt);
                tc::commit(k_empty + gt % kKStages);
                if (nkt == 1) tc::commit(q_empty);  // the unit's last S MMAs are issued
                for (int j = 0; j < nkt; ++j) {
                    if (*abort_flag) {
                        ok = false;
                        break;
                    }
                    const int g = gt + j;
                    // values of tile j; in the unit's last tile, with the rows
                    // past its keys cleared.  v_zero of a stage completes once
                    // per value tile, and the producer cannot be a stage round
                    // ahead here (it waits for v_empty of this tile), so the
                    // last tile's phase is the one this parity names.
                    ok = tc::wait_spin(v_full + g % kVStages, (g / kVStages) & 1);
                    if (ok && j == nkt - 1) ok = tc::wait_spin(v_zero + g % kVStages, (g / kVStages) & 1);
                    if (!ok) break;
                    bool kn = false;  // keys of tile j + 1 waited for
                    // Q tile A, then B: P V_X(j), then S_X(j + 1)
#pragma unroll
                    for (int X = 0; X < 2; ++X) {
                        const int ntx = X ? nt1 : nt0;
                        const int tpx = X ? tp1 : tp0;
                        if (ok && j < ntx) {
                            ok = tc::wait_spin(p_full + X, (tpx + j) & 1);
                            if (ok) {
                                tc::fence_after();
                                issue_pv(X, j, g);
                            }
                        }
                        if (ok && j + 1 < ntx) {
                            if (!kn) {
                                ok = tc::wait_spin(k_full + (g + 1) % kKStages, ((g + 1) / kKStages) & 1);
                                if (ok) tc::fence_after();
                                kn = true;
                            }
                            if (ok) issue_s(X, g + 1);
                        }
                    }
                    if (!ok) break;
                    tc::commit(v_empty + g % kVStages);
                    if (j + 1 < nkt) tc::commit(k_empty + (g + 1) % kKStages);
                    if (j + 2 == nkt) tc::commit(q_empty);  // the unit's last S MMAs are issued
                }
                if (!ok) break;
                gt += nkt;
                tp0 += nt0;
                tp1 += nt1;
            }
            if (!ok) {
                report(p.err, PKV_DEVERR_TIMEOUT);
                *abort_flag = 1;
            }
            // the tensor core is idle before the memory it uses is released
            // (a CTA whose claims all came too late issued none)
            if (any_mma) {
                tc::commit(drain);
                if (!tc::wait_spin(drain, 0)) report(p.err, PKV_DEVERR_TIMEOUT);
            }
        }
        __syncwarp();
      }
    } else {
        setmaxnreg_inc();
        // ------------------------------------------- softmax, O, epilogue
        // One thread per query row (its tensor-memory lane) of Q tile X.
        // P_j goes back into tensor memory over S_j.  S_X(j) is issued after
        // P V_X(j - 1), so when it is complete O holds every earlier tile and
        // can be rescaled without waiting.
        const int X = (warp - 4) >> 2;     // Q tile
        const int wq = warp & 3;           // tensor-memory lane quarter
        const int row = wq * 32 + lane;
        const int rq = row / G, g = row - rq * G;
        const uint32_t lane_base = static_cast<uint32_t>(wq * 32) << 16;
        const uint32_t tS = tmem + X * kTileN + lane_base;
        const uint32_t tO = tmem + 256 + X * kTileN + lane_base;
        const float c = p.qk_scale;
        const float2 c2 = make_float2(c, c);
        bool ok = true;
        int tp = 0;  // tiles of this Q tile in the finished units
        for (int k = 0;; ++k) {
            Unit u;
            const int r = next_unit(k, true, u);
            ok = r >= 0;
            if (r <= 0) break;
            const int h = u.h;
            const int ntx = ((X ? u.kv_end[1] : u.kv_end[0]) + kTileN - 1) / kTileN;
            bool row_valid;
            int pos;  // last key this row attends to
            if constexpr (!kPrefix) {
                const int tx = u.t0 + X * RQ;
                row_valid = tx + rq < u.n;
                pos = u.ctx + tx + min(rq, max(u.n - 1 - tx, 0));  // padding rows reuse the last position
            } else {
                row_valid = mrow0 + X * RQ + rq < members;
                pos = u.kv_end[0] - 1;
            }
            // prefix pass: this row's batch row, read now so the epilogue
            // does not wait for it
            const int member_row =
                kPrefix && row_valid ? __ldg(p.group_members + m0 + mrow0 + X * RQ + rq) : -1;
            float m_ref = -INFINITY, l = 0.f;
            for (int j = 0; j < ntx; ++j) {
                ok = warp_all(tc::wait_spin(s_full + X, (tp + j) & 1));
                if (!ok || !warp_all(*abort_flag == 0)) break;
                tc::fence_after();
                // P V_X(j - 1) is complete (it precedes S_X(j)): take its phase
                if (j > 0) ok = warp_all(tc::wait_spin(o_done + X, (tp + j - 1) & 1));
                if (!ok) break;
                uint32_t x[4][32];
#pragma unroll
                for (int q = 0; q < 4; ++q) tc::ld32(tS + q * 32, x[q]);
                tc::wait_ld();

                // masked keys -inf; row maximum of the raw scores (scale > 0
                // keeps the order)
                const int key0 = j * kTileN;
                if (key0 + kTileN - 1 > pos) {
#pragma unroll
                    for (int q = 0; q < 4; ++q)
#pragma unroll
                        for (int i = 0; i < 32; ++i)
                            if (key0 + q * 32 + i > pos) x[q][i] = __float_as_uint(-INFINITY);
                }
                float mx[4] = {-INFINITY, -INFINITY, -INFINITY, -INFINITY};
#pragma unroll
                for (int q = 0; q < 4; ++q)
#pragma unroll
                    for (int i = 0; i < 32; i += 2)
                        mx[(i >> 1) & 3] = fmax3(mx[(i >> 1) & 3], __uint_as_float(x[q][i]), __uint_as_float(x[q][i + 1]));
                const float mt = fmax3(fmax3(mx[0], mx[1], mx[2]), mx[3], -INFINITY) * c;
                const float m_new = fmaxf(m_ref, mt);
                const bool rebase = m_new > m_ref + kRebase;
                float alpha = 1.f;
                if (rebase) {
                    alpha = ex2(m_ref - m_new);  // 0 on the first tile (m_ref = -inf)
                    m_ref = m_new;
                }
                const float2 nm2 = make_float2(-m_ref, -m_ref);
                float2 ls[4] = {make_float2(0.f, 0.f), make_float2(0.f, 0.f), make_float2(0.f, 0.f), make_float2(0.f, 0.f)};
                // P as a 16-bit head (columns 0-63) and the head's rounding
                // error as a 16-bit tail (columns 64-127, S's second half,
                // already read): P V runs once on each, so the probabilities
                // keep 16 (bf16) or 22 (f16) significant bits
#pragma unroll
                for (int q = 0; q < 4; ++q) {
                    uint32_t pk[16], pl[16];
#pragma unroll
                    for (int i = 0; i < 16; ++i) {
                        float2 a = ffma2(make_float2(__uint_as_float(x[q][2 * i]), __uint_as_float(x[q][2 * i + 1])), c2, nm2);
                        a.x = ex2(a.x);
                        a.y = ex2(a.y);
                        ls[i & 3] = fadd2(ls[i & 3], a);
                        split2<kBF>(a, pk[i], pl[i]);
                    }
                    tc::st16(tS + q * 16, pk);
                    tc::st16(tS + 64 + q * 16, pl);
                }
                const float2 lt = fadd2(fadd2(ls[0], ls[1]), fadd2(ls[2], ls[3]));
                l = l * alpha + (lt.x + lt.y);
                if (j > 0 && __any_sync(0xffffffffu, rebase)) {
                    const float2 a2 = make_float2(alpha, alpha);
#pragma unroll
                    for (int q = 0; q < D / 32; ++q) {
                        uint32_t o[32];
                        tc::ld32(tO + q * 32, o);
                        tc::wait_ld();
#pragma unroll
                        for (int i = 0; i < 16; ++i) {
                            const float2 v = fmul2(make_float2(__uint_as_float(o[2 * i]), __uint_as_float(o[2 * i + 1])), a2);
                            o[2 * i] = __float_as_uint(v.x);
                            o[2 * i + 1] = __float_as_uint(v.y);
                        }
                        tc::st32(tO + q * 32, o);
                    }
                }
                tc::wait_st();
                tc::fence_before();
                __syncwarp();
                if (lane == 0) tc::arrive(p_full + X);
            }
            const bool live = ntx > 0 && ok && warp_all(*abort_flag == 0);
            if (live) ok = warp_all(tc::wait_spin(o_done + X, (tp + ntx - 1) & 1));
            if (live && ok) {
                tc::fence_after();
                const float inv = p.o_scale / l;
                if constexpr (!kPrefix) {
                    typename T::storage* orow =
                        reinterpret_cast<typename T::storage*>(p.out) +
                        (static_cast<int64_t>(u.q0 + u.t0 + X * RQ + rq) * p.Hq + h * G + g) * D;
#pragma unroll
                    for (int q = 0; q < D / 32; ++q) {
                        uint32_t o[32];
                        tc::ld32(tO + q * 32, o);
                        tc::wait_ld();
                        if (row_valid && p.out_v8) {
#pragma unroll
                            for (int v8 = 0; v8 < 2; ++v8) {
                                uint32_t w[8];
#pragma unroll
                                for (int i = 0; i < 8; ++i)
                                    w[i] = pack2<kBF>(__uint_as_float(o[16 * v8 + 2 * i]) * inv,
                                                      __uint_as_float(o[16 * v8 + 2 * i + 1]) * inv);
                                st_global_v8(orow + q * 32 + v8 * 16, w);
                            }
                        } else if (row_valid) {
#pragma unroll
                            for (int v4 = 0; v4 < 4; ++v4) {
                                uint4 w;
                                w.x = pack2<kBF>(__uint_as_float(o[8 * v4 + 0]) * inv, __uint_as_float(o[8 * v4 + 1]) * inv);
                                w.y = pack2<kBF>(__uint_as_float(o[8 * v4 + 2]) * inv, __uint_as_float(o[8 * v4 + 3]) * inv);
                                w.z = pack2<kBF>(__uint_as_float(o[8 * v4 + 4]) * inv, __uint_as_float(o[8 * v4 + 5]) * inv);
                                w.w = pack2<kBF>(__uint_as_float(o[8 * v4 + 6]) * inv, __uint_as_float(o[8 * v4 + 7]) * inv);
                                *reinterpret_cast<uint4*>(orow + q * 32 + v4 * 8) = w;
                            }
                        }
                    }
                } else {
                    // partial of this prefix partition: reference maximum (log2
                    // units), the sum relative to it, and O / l
                    const int b = member_row >= 0 && member_row < p.S ? member_row : -1;
                    const int64_t prow = (static_cast<int64_t>(b) * p.Hq + h * G + g) * p.NP + pp;
                    if (b >= 0) {
                        p.part_m[prow] = m_ref;
                        p.part_l[prow] = l;
                    }
#pragma unroll
                    for (int q = 0; q < D / 32; ++q) {
                        uint32_t o[32];
                        tc::ld32(tO + q * 32, o);
                        tc::wait_ld();
                        if (b >= 0) {
                            float4* po = reinterpret_cast<float4*>(p.part_o + prow * D + q * 32);
#pragma unroll
                            for (int v4 = 0; v4 < 8; ++v4)
                                po[v4] = make_float4(__uint_as_float(o[4 * v4]) * inv, __uint_as_float(o[4 * v4 + 1]) * inv,
                                                     __uint_as_float(o[4 * v4 + 2]) * inv,
                                                     __uint_as_float(o[4 * v4 + 3]) * inv);
                        }
                    }
                }
            } else if (!ok) {
                if (lane == 0) {
                    report(p.err, PKV_DEVERR_TIMEOUT);
                    *abort_flag = 1;
                }
            }
            tp += ntx;
            if (!ok || *abort_flag) break;
        }
    }
    tc::fence_before();
    __syncthreads();
    if (warp == 1) {
        tc::fence_after();
        tc::tmem_dealloc(tmem, 512);
    }
    if (!kPrefix && threadIdx.x == 0) {
        // the last CTA to finish puts the launch's counters back to zero
        __threadfence();
        if (atomicAdd(sched + 1, 1u) == gridDim.x - 1) {
            atomicExch(sched, 0u);
            atomicExch(sched + 1, 0u);
            __threadfence();
        }
    }
}

template <typename T, int D, bool kPrefix>
cudaError_t launch_tile(const PrefillParams& p, dim3 grid, const CUtensorMap& tq, const CUtensorMap& tk,
                        const CUtensorMap& tv, cudaStream_t st) {
    constexpr int kSmemBytes = Tile<D>::kSmemBytes;
    static std::once_flag once[kMaxDevices];
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
    cudaError_t attr = cudaSuccess;
    std::call_once(once[dev], [&] {
        attr = cudaFuncSetAttribute(prefill_tc_kernel<T, D, kPrefix>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                    kSmemBytes);
    });
    if (attr != cudaSuccess) return attr;
    if constexpr (!kPrefix) {
        // a programmatic dependent of the kernel before it on the stream
        cudaLaunchConfig_t cfg = {};
        cfg.gridDim = grid;
        cfg.blockDim = dim3(kThreads);
        cfg.dynamicSmemBytes = kSmemBytes;
        cfg.stream = st;
        cudaLaunchAttribute la[1];
        la[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
        la[0].val.programmaticStreamSerializationAllowed = 1;
        cfg.attrs = la;
        cfg.numAttrs = 1;
        const cudaError_t e = cudaLaunchKernelEx(&cfg, prefill_tc_kernel<T, D, kPrefix>, p, tq, tk, tv);
        if (e != cudaErrorNotSupported && e != cudaErrorInvalidValue) return e;
        (void)cudaGetLastError();  // a driver that refuses the attribute gets a plain launch
    }
    prefill_tc_kernel<T, D, kPrefix><<<grid, kThreads, kSmemBytes, st>>>(p, tq, tk, tv);
    return cudaGetLastError();
}

// Persistent prefill: one CTA per SM (one CTA fits an SM), or one per unit
// when there are fewer; the launch takes the next counter slot.
template <typename T>
cudaError_t launch_prefill(PrefillParams p, int D, const CUtensorMap& tq, const CUtensorMap& tk,
                           const CUtensorMap& tv, cudaStream_t st) {
    static std::atomic<uint32_t> next_slot{0};
    p.sched_slot = static_cast<int32_t>(next_slot.fetch_add(1u, std::memory_order_relaxed) % kSchedSlots);
    const int64_t units = p.work ? p.num_work : static_cast<int64_t>(p.num_qtiles) * p.S;
    const dim3 grid(static_cast<unsigned>(std::min<int64_t>(units * p.Hkv, num_sms())));
    return D == 64 ? launch_tile<T, 64, false>(p, grid, tq, tk, tv, st)
                   : launch_tile<T, 128, false>(p, grid, tq, tk, tv, st);
}

bool aligned16(const void* ptr) { return (reinterpret_cast<uintptr_t>(ptr) & 15u) == 0; }

// ------------------------------------------------------- fp8 pools: staging
// The tensor-core kind::f16 MMA takes 16-bit operands on both sides, so
// before the attention pass the blocks the batch reaches are copied out of
// an E4M3 pool into a 16-bit copy in q's type.  The copy is exact (every
// E4M3 value is also an f16 and a bf16 value); k_scale joins the score
// scale and v_scale the final 1 / l, so the scales cost no rounding of the
// cached codes.  Copy block s * MB + j holds sequence s's logical block j,
// and the copy's block table says so.
//
// Workspace: the copy's block table int32 [S][MB], then the K copy and the
// V copy, each [S * MB][Hkv][16][D] 16-bit, all on 256-byte boundaries.
struct StageLayout {
    int64_t table_off, k_off, v_off, bytes;
};

StageLayout stage_layout(int64_t S, int64_t MB, int64_t Hkv, int64_t D) {
    const auto up = [](int64_t x) { return (x + 255) / 256 * 256; };
    StageLayout l{};
    const int64_t copy = S * MB * Hkv * kBlockSize * D * 2;
    l.table_off = 0;
    l.k_off = up(S * MB * 4);
    l.v_off = l.k_off + up(copy);
    l.bytes = l.v_off + up(copy);
    return l;
}

// One CTA per (logical block j, sequence s, pool z: 0 keys, 1 values):
// converts the block's codes of every KV head.  A thread takes 8 codes (8 bytes in, one 16-byte
// vector out), so each warp reads 256 and writes 512 contiguous bytes, and it
// issues kStageUnroll loads before it converts.  Blocks at or past the
// sequence's length are skipped; a block id outside the pool is reported and
// its copy zeroed (the attention pass then reads zeros, not stale bytes).
constexpr int kStageUnroll = 8;

// kGroups = false (prefill): CTA (j, s, z) copies sequence s's logical block
// j into copy block s * MB + j, for the blocks its seq_lens[s] reaches.
// kGroups = true (cascade decode): CTA (j, g, z) copies block j of group g's
// shared prefix (group_blocks[g] blocks, read through the block table of
// the group's first member) into copy block g * MGB + j, and that member's
// row of the copy's table names it; the prefix pass reads only those rows.
template <typename T, bool kGroups>
__global__ void __launch_bounds__(256) stage_fp8_kernel(const uint8_t* __restrict__ k_cache,
                                                        const uint8_t* __restrict__ v_cache,
                                                        const int32_t* __restrict__ block_tables,
                                                        const int32_t* __restrict__ seq_lens, int MB, int NB,
                                                        int block_vecs, uint4* __restrict__ k_copy,
                                                        uint4* __restrict__ v_copy, int32_t* __restrict__ table_copy,
                                                        unsigned int* err, const int32_t* __restrict__ group_blocks,
                                                        const int32_t* __restrict__ group_offsets,
                                                        const int32_t* __restrict__ group_members, int S, int MGB) {
    constexpr bool kBF = std::is_same<T, BF16>::value;
    // the attention kernel may start its setup once every CTA here has begun
    allow_dependent_launch();
    const int j = blockIdx.x, z = blockIdx.z;
    int64_t row, dst;  // table entry read (and written in the copy), copy block
    if constexpr (kGroups) {
        const int g = blockIdx.y;
        const int nb = min(max(__ldg(group_blocks + g), 0), MB);  // the prefix pass reports a bad count
        const int s0 = __ldg(group_members + __ldg(group_offsets + g));
        if (j >= nb || s0 < 0 || s0 >= S) return;  // ... and a bad member
        row = static_cast<int64_t>(s0) * MB + j;
        dst = static_cast<int64_t>(g) * MGB + j;
    } else {
        const int s = blockIdx.y;
        const int L = __ldg(seq_lens + s);  // the attention pass reports a bad length
        const int nblk = L <= 0 ? 0 : min((L + kBlockSize - 1) / kBlockSize, MB);
        if (j >= nblk) return;
        row = static_cast<int64_t>(s) * MB + j;
        dst = row;
    }
    const int id = __ldg(block_tables + row);
    const bool bad = id < 0 || id >= NB;
    if (threadIdx.x == 0 && z == 0) {
        table_copy[row] = static_cast<int32_t>(dst);
        if (bad) report(err, PKV_DEVERR_BLOCK_ID);
    }
    // block_vecs: 16-byte output vectors per block and pool (Hkv * 16 * D / 8)
    const int64_t src = static_cast<int64_t>(bad ? 0 : id) * block_vecs;
    const uint2* sp = reinterpret_cast<const uint2*>(z ? v_cache : k_cache) + src;
    uint4* dp = (z ? v_copy : k_copy) + dst * block_vecs;
    const int total = block_vecs;
    for (int base = 0; base < total; base += kStageUnroll * blockDim.x) {
        uint2 w[kStageUnroll];
#pragma unroll
        for (int u = 0; u < kStageUnroll; ++u) {
            const int i = base + u * blockDim.x + threadIdx.x;
            w[u] = make_uint2(0u, 0u);
            if (i < total && !bad) w[u] = __ldcs(sp + i);  // read once
        }
#pragma unroll
        for (int u = 0; u < kStageUnroll; ++u) {
            const int i = base + u * blockDim.x + threadIdx.x;
            if (i >= total) continue;
            const uint32_t words[2] = {w[u].x, w[u].y};
            float f[8];
            Unpack<E4M3, 8>::run(words, f);
            uint4 o;
            o.x = pack2<kBF>(f[0], f[1]);
            o.y = pack2<kBF>(f[2], f[3]);
            o.z = pack2<kBF>(f[4], f[5]);
            o.w = pack2<kBF>(f[6], f[7]);
            dp[i] = o;
        }
    }
}

}  // namespace

int prefix_partitions(int blocks) { return (blocks + kPrefixPartitionBlocks - 1) / kPrefixPartitionBlocks; }

cudaError_t launch_cascade_prefix_tc(const CascadeParams& cp, int num_groups, int q_dtype, int D, const CUtensorMap& tq,
                                     const CUtensorMap& tk, const CUtensorMap& tv, cudaStream_t st) {
    const DecodeParams& b = cp.base;
    PrefillParams p{};
    p.block_tables = cp.prefix_tables;
    p.S = b.S;
    p.Hq = b.Hq;
    p.Hkv = b.Hkv;
    p.MB = b.MB;
    p.NB = cp.prefix_nb;
    p.G = cp.G;
    p.TT = kTileM / cp.G;
    p.qk_scale = cp.prefix_qk_scale;
    p.o_scale = cp.prefix_o_scale;
    p.err = b.err;
    p.group_offsets = cp.group_offsets;
    p.group_members = cp.group_members;
    p.group_blocks = b.group_blocks;
    p.part_m = b.part_m;
    p.part_l = b.part_l;
    p.part_o = b.part_o;
    p.NP = b.NP;
    p.row_chunks = cp.row_chunks;
    const dim3 grid(cp.npp, b.Hkv, num_groups * cp.row_chunks);
    if (q_dtype == PKV_BF16)
        return D == 64 ? launch_tile<BF16, 64, true>(p, grid, tq, tk, tv, st)
                       : launch_tile<BF16, 128, true>(p, grid, tq, tk, tv, st);
    return D == 64 ? launch_tile<F16, 64, true>(p, grid, tq, tk, tv, st)
                   : launch_tile<F16, 128, true>(p, grid, tq, tk, tv, st);
}

CascadeStage cascade_stage_layout(int64_t S, int64_t MB, int64_t num_groups, int64_t MGB, int64_t Hkv, int64_t D) {
    const auto up = [](int64_t x) { return (x + 255) / 256 * 256; };
    const int64_t copy = num_groups * MGB * Hkv * kBlockSize * D * 2;
    CascadeStage l{};
    l.table_off = 0;
    l.k_off = up(S * MB * 4);
    l.v_off = l.k_off + up(copy);
    l.bytes = l.v_off + up(copy);
    return l;
}

cudaError_t launch_cascade_stage_fp8(const CascadeParams& cp, int num_groups, int MGB, int q_dtype,
                                     const void* k_cache, const void* v_cache, void* staging, cudaStream_t st) {
    const DecodeParams& b = cp.base;
    if (num_groups == 0 || MGB == 0) return cudaSuccess;
    const CascadeStage lay = cascade_stage_layout(b.S, b.MB, num_groups, MGB, b.Hkv, b.D);
    unsigned char* ws = static_cast<unsigned char*>(staging);
    int32_t* table_copy = reinterpret_cast<int32_t*>(ws + lay.table_off);
    uint4* k_copy = reinterpret_cast<uint4*>(ws + lay.k_off);
    uint4* v_copy = reinterpret_cast<uint4*>(ws + lay.v_off);
    const int block_vecs = b.Hkv * kBlockSize * b.D / 8;
    const dim3 grid(static_cast<unsigned>(MGB), static_cast<unsigned>(num_groups), 2);
    const auto* kc = static_cast<const uint8_t*>(k_cache);
    const auto* vc = static_cast<const uint8_t*>(v_cache);
    if (q_dtype == PKV_BF16)
        stage_fp8_kernel<BF16, true><<<grid, 256, 0, st>>>(kc, vc, b.block_tables, b.seq_lens, b.MB, b.NB, block_vecs,
                                                           k_copy, v_copy, table_copy, b.err, b.group_blocks,
                                                           cp.group_offsets, cp.group_members, b.S, MGB);
    else
        stage_fp8_kernel<F16, true><<<grid, 256, 0, st>>>(kc, vc, b.block_tables, b.seq_lens, b.MB, b.NB, block_vecs,
                                                          k_copy, v_copy, table_copy, b.err, b.group_blocks,
                                                          cp.group_offsets, cp.group_members, b.S, MGB);
    return cudaGetLastError();
}

}  // namespace pkv

using namespace pkv;

extern "C" pkv_status pkv_paged_attention_prefill(const void* q, int32_t q_dtype, int32_t num_tokens,
                                                  int32_t num_q_heads, int32_t num_seqs, const int32_t* query_start,
                                                  int32_t max_query_len, const void* k_cache, const void* v_cache,
                                                  const pkv_cache_desc* desc, const int32_t* block_tables,
                                                  int32_t max_blocks_per_seq, const int32_t* seq_lens,
                                                  const int32_t* work_units, int32_t num_work_units, float scale,
                                                  void* out, void* workspace, size_t workspace_bytes,
                                                  void* stream) {
    if (!desc || num_tokens < 0 || num_seqs < 0 || max_query_len < 0 || num_q_heads <= 0) return PKV_ERR_INVALID;
    if (num_work_units < 0 || (!work_units && num_work_units > 0)) return PKV_ERR_INVALID;
    if (desc->block_size != kBlockSize || desc->num_kv_heads <= 0 || desc->num_blocks <= 0) return PKV_ERR_INVALID;
    if (num_q_heads % desc->num_kv_heads) return PKV_ERR_INVALID;
    const int G = num_q_heads / desc->num_kv_heads;
    const int D = desc->head_size;
    if ((D != 64 && D != 128) || (G != 1 && G != 2 && G != 4 && G != 8)) return PKV_ERR_UNSUPPORTED;
    const bool fp8 = desc->kv_dtype == PKV_FP8_E4M3;
    if (desc->kv_dtype != PKV_F16 && desc->kv_dtype != PKV_BF16 && !fp8) return PKV_ERR_UNSUPPORTED;
    if (fp8 ? (q_dtype != PKV_F16 && q_dtype != PKV_BF16) : q_dtype != desc->kv_dtype) return PKV_ERR_UNSUPPORTED;
    if (!(scale > 0.f) || scale > 3.0e38f) return PKV_ERR_INVALID;  // finite, > 0 (max on raw scores)
    if (fp8 && !(desc->k_scale > 0.f && desc->k_scale < 3.0e38f && desc->v_scale > 0.f && desc->v_scale < 3.0e38f))
        return PKV_ERR_INVALID;
    if (fp8 && !(scale * desc->k_scale < 3.0e38f)) return PKV_ERR_INVALID;
    if (num_seqs == 0 || num_tokens == 0 || max_query_len == 0 || (work_units && num_work_units == 0)) return PKV_OK;
    if (!q || !out || !k_cache || !v_cache || !block_tables || !seq_lens || !query_start) return PKV_ERR_INVALID;
    if (max_blocks_per_seq <= 0 || !aligned16(q) || !aligned16(out) || !aligned16(k_cache) || !aligned16(v_cache))
        return PKV_ERR_INVALID;
    if (num_seqs > 65535 || desc->num_kv_heads > 65535) return PKV_ERR_UNSUPPORTED;
    if (static_cast<int64_t>(desc->num_blocks) * desc->num_kv_heads * kBlockSize > INT32_MAX) return PKV_ERR_UNSUPPORTED;
    StageLayout lay{};
    if (fp8) {
        // the copy is a pool of num_seqs * max_blocks_per_seq blocks
        if (static_cast<int64_t>(num_seqs) * max_blocks_per_seq * desc->num_kv_heads * kBlockSize > INT32_MAX)
            return PKV_ERR_UNSUPPORTED;
        lay = stage_layout(num_seqs, max_blocks_per_seq, desc->num_kv_heads, D);
        if (!workspace || static_cast<int64_t>(workspace_bytes) < lay.bytes) return PKV_ERR_WORKSPACE;
        if (!aligned16(workspace)) return PKV_ERR_INVALID;
    }
    unsigned int* err = error_word();
    if (!err) return PKV_ERR_CUDA;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    const void* k_pool = k_cache;
    const void* v_pool = v_cache;
    int32_t pool_blocks = desc->num_blocks;
    if (fp8) {
        uint8_t* ws = static_cast<uint8_t*>(workspace);
        int32_t* table_copy = reinterpret_cast<int32_t*>(ws + lay.table_off);
        uint4* k_copy = reinterpret_cast<uint4*>(ws + lay.k_off);
        uint4* v_copy = reinterpret_cast<uint4*>(ws + lay.v_off);
        const int block_vecs = desc->num_kv_heads * kBlockSize * D / 8;  // 8 codes -> one 16-byte vector
        const dim3 grid(static_cast<unsigned>(max_blocks_per_seq), static_cast<unsigned>(num_seqs), 2);
        const auto* kc = static_cast<const uint8_t*>(k_cache);
        const auto* vc = static_cast<const uint8_t*>(v_cache);
        if (q_dtype == PKV_BF16)
            stage_fp8_kernel<BF16, false><<<grid, 256, 0, st>>>(kc, vc, block_tables, seq_lens, max_blocks_per_seq,
                                                                desc->num_blocks, block_vecs, k_copy, v_copy,
                                                                table_copy, err, nullptr, nullptr, nullptr, 0, 0);
        else
            stage_fp8_kernel<F16, false><<<grid, 256, 0, st>>>(kc, vc, block_tables, seq_lens, max_blocks_per_seq,
                                                               desc->num_blocks, block_vecs, k_copy, v_copy,
                                                               table_copy, err, nullptr, nullptr, nullptr, 0, 0);
        if (cudaGetLastError() != cudaSuccess) return PKV_ERR_CUDA;
        block_tables = table_copy;
        k_pool = k_copy;
        v_pool = v_copy;
        pool_blocks = num_seqs * max_blocks_per_seq;
    }

    PrefillParams p{};
    p.query_start = query_start;
    p.block_tables = block_tables;
    p.seq_lens = seq_lens;
    p.out = out;
    p.S = num_seqs;
    p.T = num_tokens;
    p.Hq = num_q_heads;
    p.Hkv = desc->num_kv_heads;
    p.MB = max_blocks_per_seq;
    p.NB = pool_blocks;
    p.G = G;
    p.TT = kTileM / G;
    p.num_qtiles = (max_query_len + 2 * p.TT - 1) / (2 * p.TT);  // CTAs of two Q tiles
    if (static_cast<int64_t>(p.num_qtiles) * p.Hkv * p.S > INT32_MAX) return PKV_ERR_UNSUPPORTED;  // one grid axis
    p.work = work_units;
    p.num_work = num_work_units;
    if (static_cast<int64_t>(num_work_units) * p.Hkv > INT32_MAX) return PKV_ERR_UNSUPPORTED;
    p.max_query_len = max_query_len;
    p.qk_scale = scale * (fp8 ? desc->k_scale : 1.f) * 1.4426950408889634f;
    p.o_scale = fp8 ? desc->v_scale : 1.f;
    p.out_v8 = (reinterpret_cast<uintptr_t>(out) & 31u) == 0;  // rows are multiples of 128 bytes
    p.err = err;

    CUtensorMap tq, tk, tv;
    const int64_t pool_rows = static_cast<int64_t>(pool_blocks) * desc->num_kv_heads * kBlockSize;
    if (!encode_token_head_map(&tq, q, D, num_q_heads, num_tokens, G, kTileM / G) ||
        !encode_pool_map(&tk, k_pool, 2, pool_rows, D) || !encode_pool_map(&tv, v_pool, 2, pool_rows, D))
        return PKV_ERR_CUDA;
    const cudaError_t e = q_dtype == PKV_BF16 ? launch_prefill<BF16>(p, D, tq, tk, tv, st)
                                              : launch_prefill<F16>(p, D, tq, tk, tv, st);
    return e == cudaSuccess ? PKV_OK : PKV_ERR_CUDA;
}

extern "C" size_t pkv_prefill_workspace_bytes(int32_t kv_dtype, int32_t num_seqs, int32_t num_kv_heads,
                                              int32_t head_size, int32_t max_blocks_per_seq) {
    if (num_seqs < 0 || num_kv_heads <= 0 || head_size <= 0 || max_blocks_per_seq < 0) return 0;
    if (kv_dtype != PKV_FP8_E4M3) return 0;  // 16-bit pools are read in place
    return static_cast<size_t>(stage_layout(num_seqs, max_blocks_per_seq, num_kv_heads, head_size).bytes);
}
