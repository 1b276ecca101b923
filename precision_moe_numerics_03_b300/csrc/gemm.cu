// gemm.cu -- block-scaled grouped expert GEMMs on the 5th-generation tensor cores (tcgen05).
//
// Method: the forward pass of the expert layers runs in NVFP4 with a dedicated kernel, the
// backward pass in MXFP8 ("Inkling 2 Small's Native 4-Bit Training: Debut and Doubts",
// agihunt.info, "Confirmed"; "Thinking Machines: Nvidia FP4 Up to 6x Faster, Runs Gain 8%",
// fourweekmba.com, "What Thinking Machines Changed").
//
// One persistent CTA per SM, 12 warps:
//   warp 0 (one lane)  TMA producer: A tile 128 rows x 128 bytes, B tile 256 rows x 128 bytes
//                      (128-byte swizzle), and the two tiles' scale factors (1-D bulk copies of
//                      the tensor-core scale layout), into a 4-stage shared-memory ring;
//   warp 1 (one lane)  MMA issuer: per stage, tcgen05.cp of the scale factors into tensor memory,
//                      then four tcgen05.mma (kind::mxf4nvf4 with 4 UE4M3 scales per 64 values, or
//                      kind::mxf8f6f4 E4M3 with one UE8M0 scale per 32), accumulating a 128x256
//                      binary32 tile in tensor memory; tcgen05.commit frees the stage;
//   warp 2             allocates / frees the 512 tensor-memory columns;
//   warps 4..11        epilogue: tcgen05.ld of the accumulator (warp w reads lanes 32*(w%4).. and
//                      half (w-4)/4 of the columns), times the per-tensor scales, to binary32 or
//                      bf16 in global memory, added into binary32, or (the fused weight-gradient
//                      mode) applied as an SGD step to FP32 master weights with their bf16 copy
//                      and per-expert amax written on the way.
// Every mbarrier wait is bounded (about two seconds of SM clock); a wait that gives up sets the
// library status word, stops the CTA's loops, drains its own copies and MMAs, and frees tensor
// memory before the CTA exits.

#include "common.cuh"

#include <cuda.h>
#include <cudaTypedefs.h>

namespace moe4 {

__device__ unsigned int g_status = 0;

namespace gemm {

constexpr int BM = 128;         // rows of A per tile (MMA M)
constexpr int BN = 256;         // rows of B per tile (MMA N); the fused SGD mode uses 128
constexpr int BKB = 128;        // bytes of contraction per stage (one 128-byte swizzle row)
constexpr int STAGES = 4;
constexpr int THREADS = 384;    // warps 0..3: producer, MMA, TMEM, spare; 4..11: epilogue
constexpr int EPI_THREADS = 256;
constexpr int A_TILE = BM * BKB;
constexpr int TMEM_COLS = 512;
constexpr long long kWaitCycles = 1ll << 32;

template <int KIND>
struct Cfg;
template <>
struct Cfg<0> {                       // NVFP4
    static constexpr int ELEMS = 256;  // contraction elements per stage
    static constexpr int ATOMS = 4;    // 512-byte scale atoms per 128-row tile per stage
    static constexpr int ELEMS_PER_ATOM = 64;
};
template <>
struct Cfg<1> {                       // MXFP8
    static constexpr int ELEMS = 128;
    static constexpr int ATOMS = 1;
    static constexpr int ELEMS_PER_ATOM = 128;
};

// Epilogue staging of the fused SGD mode, per epilogue warp: a ring of buffers, each a 32x16
// binary32 chunk (64-byte rows, 64-byte swizzle) and, when the bf16 copy is written, a 32x16 bf16
// chunk (32-byte rows, 32-byte swizzle), with one mbarrier per buffer.  Master-weight loads run a
// fixed number of chunks ahead of the chunk being updated, so each warp keeps several loads in
// flight; without the bf16 chunks the ring has room to run further ahead (SgdRing below).
constexpr int SGD_CW = 16;                    // columns per chunk
constexpr int SGD_W_CHUNK = 32 * SGD_CW * 4;  // 2 KB
constexpr int SGD_B_CHUNK = 32 * SGD_CW * 2;  // 1 KB
// TMA-store epilogue: one staged chunk of 32 rows per epilogue warp, TMA_CW columns wide (32 for
// NVFP4; 16 for MXFP8, whose smaller staging leaves room for a fourth operand stage)
template <int KIND>
constexpr int TMA_CW = KIND == 0 ? 32 : 16;
template <int KIND>
constexpr int EPI_W_TILE = 32 * TMA_CW<KIND> * 4;
// Epilogue implementations: REG stores from registers (the read-modify-write accumulate mode),
// TMA stages each warp's 32x32 output tile in shared memory and bulk-stores it, SGD is the fused
// master-weight update.  Operand stages shrink to make room for the staging buffers.
// SWI (the gate/up projection, NVFP4): each tile's 256 B rows are 128 gate rows and the matching
// 128 up rows, so the epilogue holds gate and up of the same columns and writes GU and the SwiGLU
// h = silu(g) * u (bf16) with its amax, as TMA does for D.
// SWB (the down projection's dgrad, MXFP8): the epilogue applies the SwiGLU backward to the product
// dH, reading GU through a two-chunk ring per warp and writing dGU (bf16); dH is not stored.
enum EpiImpl : int { EPI_REG = 0, EPI_TMA = 1, EPI_SGD = 2, EPI_HMX = 3, EPI_SGD32 = 4, EPI_SWI = 5, EPI_SWB = 6 };
// EPI_SWB ring, per epilogue warp: two buffers, each the gate and the up 32x16 binary32 chunk of
// GU (64-byte rows, 64-byte swizzle); dg and du (32x16 bf16, 32-byte rows) are written over the
// gate chunk and stored from there.
constexpr int SWB_BUF = 4096;
constexpr int SWB_WARP_BYTES = 2 * SWB_BUF;
// EPI_SGD writes the bf16 copy, EPI_SGD32 only the binary32 master weights (and the amax).
__host__ __device__ constexpr bool is_sgd(int em) { return em == EPI_SGD || em == EPI_SGD32; }
template <int EM>
struct SgdRing {
    static constexpr bool BF16 = EM == EPI_SGD;
    static constexpr int NB = BF16 ? 3 : 5;  // ring buffers per warp
    static constexpr int LA = BF16 ? 1 : 3;  // load lookahead, chunks
    static constexpr int B_CHUNK = BF16 ? SGD_B_CHUNK : 0;
    static constexpr int WARP_BYTES = NB * (SGD_W_CHUNK + B_CHUNK);
    // the store that last read a refilled buffer may still be the one pending group allowed
    static_assert(LA == NB - 2, "bulk_wait_read_1 before a refill assumes LA = NB - 2");
};
constexpr int SGD_NB_MAX = 5;
// Fused return-path codec (NVFP4 GEMM): each epilogue warp stages its 32 rows x 128 columns of
// bf16 product (rows padded to 272 bytes: conflict-free 16-byte stores and loads).
constexpr int HMX_PITCH = 128 * 2 + 16;
constexpr int HMX_WARP_BYTES = 32 * HMX_PITCH;
constexpr int EPI_HMX_BYTES = 8 * HMX_WARP_BYTES;
template <int KIND>
constexpr int EPI_TMA_BYTES = 8 * EPI_W_TILE<KIND>;
template <int EM>
struct EpiCfg {
    // fused SGD: 128-column tiles, so three binary32 accumulators fit in tensor memory and a
    // tile's MMAs overlap the two previous tiles' master-weight traffic
    static constexpr int BNT = is_sgd(EM) ? 128 : BN;
    static constexpr int NST =
        is_sgd(EM) ? 4 : ((EM == EPI_TMA || EM == EPI_SWI || EM == EPI_SWB) ? 3 : (EM == EPI_HMX ? 2 : STAGES));
    // operand stages for a given operand kind: the MXFP8 TMA-store mode fits a fourth one
    template <int KIND>
    static constexpr int NSTK = (EM == EPI_TMA && KIND == 1) ? 4 : NST;
    template <int KIND>
    static constexpr int BYTESK =
        is_sgd(EM) ? 8 * SgdRing<EM>::WARP_BYTES
                   : ((EM == EPI_TMA || EM == EPI_SWI) ? EPI_TMA_BYTES<KIND>
                                                       : (EM == EPI_HMX ? EPI_HMX_BYTES
                                                                        : (EM == EPI_SWB ? 8 * SWB_WARP_BYTES : 0)));
};

template <int KIND, int NST, int EPI, int BNT>
struct Layout {
    static constexpr int RT = BNT / 128;  // 128-row tiles of B per tile
    static constexpr int B_TILE = BNT * BKB;
    static constexpr int SFA = Cfg<KIND>::ATOMS * 512;
    static constexpr int SFB = RT * Cfg<KIND>::ATOMS * 512;
    static constexpr int OFF_A = 0;
    static constexpr int OFF_B = OFF_A + NST * A_TILE;
    static constexpr int OFF_SFA = OFF_B + NST * B_TILE;
    static constexpr int OFF_SFB = OFF_SFA + NST * SFA;
    static constexpr int OFF_EPI = (OFF_SFB + NST * SFB + 1023) / 1024 * 1024;
    static constexpr int OFF_BAR = OFF_EPI + EPI;
    // full, empty, tmem_full[3], tmem_empty[3], drain, epilogue
    static constexpr int NBAR = 2 * NST + 7 + 8 * SGD_NB_MAX;
    static constexpr int OFF_MISC = OFF_BAR + NBAR * 8;
    static constexpr int BYTES = OFF_MISC + 16;
    static constexpr int SMEM = BYTES + 1024;    // room to align the base to 1024
    static constexpr int TX = A_TILE + B_TILE + SFA + SFB;
    // tensor-memory columns: NACC accumulators of BNT columns, then per stage SFA and SFB
    static constexpr int SF_COLS_A = Cfg<KIND>::ATOMS * 4;
    static constexpr int SF_COLS_B = Cfg<KIND>::ATOMS * 4 * RT;
    static constexpr int SF_COLS = SF_COLS_A + SF_COLS_B;
    // three accumulators where they fit (the fused SGD's 128-column tiles): the MMAs of a long
    // contraction can then start while the epilogue still streams two earlier tiles' weights
    static constexpr int NACC = (BNT == 128 && 3 * BNT + NST * SF_COLS <= TMEM_COLS)
                                    ? 3
                                    : (2 * BNT + NST * SF_COLS <= TMEM_COLS ? 2 : 1);
    static constexpr int SF_BASE = NACC * BNT;
    static_assert(SF_BASE + NST * SF_COLS <= TMEM_COLS, "tensor memory overflow");
    static_assert(SMEM <= 232448, "shared memory overflow");
};

enum Out : int { F32 = 0, BF16 = 1, ACC_F32 = 2, SGD = 3 };

struct Args {
    const uint8_t *sfa;     // tensor-core scale layout of A
    const uint8_t *sfb;     // tensor-core scale layout of B
    const float *a_g_dec;   // NVFP4 only
    const float *b_g_dec;   // NVFP4 only, [E]
    const int32_t *offs;    // [E+1]
    int E;
    int group_k;            // 0: groups are row ranges of A/D; 1: ranges of the contraction
    int64_t M, N, K;        // D is [M, N] per group (group_k: [E, M, N]); K = contraction length
    void *d;
    int mode;               // Out::*
    uint16_t *w_bf16;       // Out::Sgd: the bf16 copy of the updated weights
    float lr;               // Out::Sgd
    unsigned int *amax;     // Out::Sgd: per-expert max |bf16 copy| as binary32 bits
    uint8_t *e8;            // fused codec: E8M0 scales [M, N/32] (d holds the E4M3 codes [M, N])
    unsigned int *had_amax; // bf16 output: max |Hadamard(128)-rotated rows| (binary32 bits), or null
    const int32_t *order;   // contraction-grouped: experts by decreasing group size, or null
    int64_t swiglu_f;       // EPI_SWI: the SwiGLU width f (B = W_gu [E, 2f, K]; tiles step 128 columns of f)
    int64_t swb_f;          // EPI_SWB: f (GU and dGU are [M, 2f]; the up half starts at column f)
    uint16_t *h;            // EPI_SWI: h [M, f] bf16
    unsigned int *h_amax;   // EPI_SWI: max |h| as binary32 bits
    int64_t num_tiles;
    int n_tiles_n, n_tiles_m;
    int64_t sfa_tile_stride;  // atoms between consecutive 128-row tiles of A's scale layout
    int64_t sfb_tile_stride;
};

// ------------------------------------------------------------------ PTX wrappers
__device__ __forceinline__ uint32_t smem_u32(const void *p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}
__device__ __forceinline__ void mbar_init(uint64_t *bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count) : "memory");
}
__device__ __forceinline__ void mbar_expect_tx(uint64_t *bar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)), "r"(bytes)
                 : "memory");
}
__device__ __forceinline__ void mbar_arrive(uint64_t *bar) {
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
}
__device__ __forceinline__ bool mbar_try_wait(uint32_t bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n"
        ".reg .pred p;\n"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n"
        "selp.u32 %0, 1, 0, p;\n"
        "}"
        : "=r"(ok)
        : "r"(bar), "r"(parity)
        : "memory");
    return ok != 0;
}
// Bounded wait: false when the CTA is aborting or the wait ran out (which starts the abort).
// Waits for the phase of `parity` to complete, at most `limit` SM clock cycles; on expiry it
// raises the CTA's abort flag and the library status word (reported by moe4_get_status).
__device__ __forceinline__ bool mbar_wait(uint64_t *bar, uint32_t parity, volatile int *abort_flag,
                                          long long limit = kWaitCycles) {
    const uint32_t a = smem_u32(bar);
    if (mbar_try_wait(a, parity)) return true;
    const long long t0 = clock64();
    while (true) {
#pragma unroll 1
        for (int i = 0; i < 32; ++i)
            if (mbar_try_wait(a, parity)) return true;
        if (*abort_flag) return false;
        if (clock64() - t0 > limit) {
            *abort_flag = 1;
            atomicOr(&g_status, 1u);
            return false;
        }
    }
}
__device__ __forceinline__ void tma_load_2d(void *dst, const CUtensorMap *map, uint64_t *bar, int x, int y) {
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1, {%3, %4}], [%2];" ::"r"(
            smem_u32(dst)),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(smem_u32(bar)), "r"(x), "r"(y)
        : "memory");
}
__device__ __forceinline__ void tma_store_2d(const CUtensorMap *map, const void *src, int x, int y) {
    asm volatile("cp.async.bulk.tensor.2d.global.shared::cta.bulk_group [%0, {%2, %3}], [%1];" ::"l"(
                     reinterpret_cast<uint64_t>(map)),
                 "r"(smem_u32(src)), "r"(x), "r"(y)
                 : "memory");
}
__device__ __forceinline__ void bulk_commit() { asm volatile("cp.async.bulk.commit_group;" ::: "memory"); }
__device__ __forceinline__ void bulk_wait_read_all() { asm volatile("cp.async.bulk.wait_group.read 0;" ::: "memory"); }
__device__ __forceinline__ void bulk_wait_read_1() { asm volatile("cp.async.bulk.wait_group.read 1;" ::: "memory"); }
__device__ __forceinline__ void bulk_wait_all() { asm volatile("cp.async.bulk.wait_group 0;" ::: "memory"); }
__device__ __forceinline__ void fence_async_smem() { asm volatile("fence.proxy.async.shared::cta;" ::: "memory"); }
__device__ __forceinline__ void bulk_load(void *dst, const void *src, uint32_t bytes, uint64_t *bar) {
    asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
                     smem_u32(dst)),
                 "l"(src), "r"(bytes), "r"(smem_u32(bar))
                 : "memory");
}
__device__ __forceinline__ void tc_fence_before() { asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void tc_fence_after() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void tc_commit(uint64_t *bar) {
    asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(smem_u32(bar))
                 : "memory");
}
__device__ __forceinline__ void tc_cp_sf(uint32_t taddr, uint64_t sdesc) {
    asm volatile("tcgen05.cp.cta_group::1.32x128b.warpx4 [%0], %1;" ::"r"(taddr), "l"(sdesc) : "memory");
}
template <int KIND>
__device__ __forceinline__ void tc_mma(uint32_t d, uint64_t adesc, uint64_t bdesc, uint32_t idesc, uint32_t sfa,
                                       uint32_t sfb, uint32_t accumulate) {
    if constexpr (KIND == 0) {
        asm volatile(
            "{\n"
            ".reg .pred p;\n"
            "setp.ne.u32 p, %6, 0;\n"
            "tcgen05.mma.cta_group::1.kind::mxf4nvf4.block_scale.scale_vec::4X [%0], %1, %2, %3, [%4], [%5], p;\n"
            "}" ::"r"(d),
            "l"(adesc), "l"(bdesc), "r"(idesc), "r"(sfa), "r"(sfb), "r"(accumulate)
            : "memory");
    } else {
        asm volatile(
            "{\n"
            ".reg .pred p;\n"
            "setp.ne.u32 p, %6, 0;\n"
            "tcgen05.mma.cta_group::1.kind::mxf8f6f4.block_scale.scale_vec::1X [%0], %1, %2, %3, [%4], [%5], p;\n"
            "}" ::"r"(d),
            "l"(adesc), "l"(bdesc), "r"(idesc), "r"(sfa), "r"(sfb), "r"(accumulate)
            : "memory");
    }
}
__device__ __forceinline__ void tc_ld32(uint32_t taddr, uint32_t (&r)[32]) {
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, "
        "%15, %16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31}, [%32];"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]), "=r"(r[8]),
          "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15]), "=r"(r[16]),
          "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]),
          "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
        : "r"(taddr)
        : "memory");
    asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
}

// The same load without the wait (several loads, then one tc_wait_ld).
__device__ __forceinline__ void tc_ld32_nw(uint32_t taddr, uint32_t *r) {
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, "
        "%15, %16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31}, [%32];"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]), "=r"(r[8]),
          "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15]), "=r"(r[16]),
          "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]),
          "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
        : "r"(taddr)
        : "memory");
}
__device__ __forceinline__ void tc_wait_ld() { asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory"); }

__device__ __forceinline__ void tc_ld16(uint32_t taddr, uint32_t (&r)[16]) {
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, "
        "%15}, [%16];"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]), "=r"(r[8]),
          "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15])
        : "r"(taddr)
        : "memory");
    asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
}

// Shared-memory matrix descriptor: start address, leading / stride byte offsets (16-byte units),
// the fixed version bit 46, and the swizzle mode in bits 61..63 (2 = 128-byte, 0 = none).
__device__ __forceinline__ uint64_t smem_desc(uint32_t addr, uint32_t lbo, uint32_t sbo, uint32_t swizzle) {
    return (uint64_t)((addr >> 4) & 0x3FFFu) | ((uint64_t)((lbo >> 4) & 0x3FFFu) << 16) |
           ((uint64_t)((sbo >> 4) & 0x3FFFu) << 32) | (1ull << 46) | ((uint64_t)swizzle << 61);
}

// Instruction descriptor of the block-scaled kinds: B scale id [4,6), A format [7,10), B format
// [10,13), K-major A and B (bits 15, 16 clear), N>>3 [17,23), scale type bit 23 (0 UE4M3,
// 1 UE8M0), M>>4 [24,29), A scale id [29,31).
template <int KIND, int BNT>
__device__ __forceinline__ uint32_t make_idesc(uint32_t sf_id) {
    const uint32_t fmt = KIND == 0 ? 1u : 0u;       // E2M1 for mxf4nvf4, E4M3 for mxf8f6f4
    const uint32_t scale_type = KIND == 0 ? 0u : 1u;
    return (sf_id << 4) | (fmt << 7) | (fmt << 10) | ((uint32_t)(BNT >> 3) << 17) | (scale_type << 23) |
           ((uint32_t)(BM >> 4) << 24) | (sf_id << 29);
}

struct Tile {
    int64_t m0, n0;     // first row of A / D, first row of B (N index)
    int64_t b_row;      // first row of B in the B tensor (expert offset folded in)
    int64_t k_begin;    // contraction start (elements)
    int n_stages;
    int e;
};

template <int KIND, int BNT>
__device__ __forceinline__ Tile decode_tile(const Args &p, int64_t t, int64_t ntiles) {
    Tile tl;
    // tile indices and counts are below 2^31: 32-bit division (the 64-bit one is a long sequence)
    const uint32_t t32 = (uint32_t)t, ntn = (uint32_t)p.n_tiles_n;
    if (!p.group_k) {
        const uint32_t mt = t32 / ntn, nt = t32 - mt * ntn;
        tl.m0 = (int64_t)mt * BM;
        tl.n0 = (int64_t)nt * (p.swiglu_f ? 128 : BNT);  // SwiGLU: the tile's gate columns n0 .. n0 + 127
        int lo = 0, hi = p.E;  // largest e with offs[e] <= m0
        while (hi - lo > 1) {
            const int mid = (lo + hi) >> 1;
            if (__ldg(p.offs + mid) <= tl.m0) lo = mid; else hi = mid;
        }
        tl.e = lo;
        tl.b_row = (int64_t)lo * p.N + tl.n0;
        tl.k_begin = 0;
        tl.n_stages = (int)(p.K / Cfg<KIND>::ELEMS);
    } else {
        // With an expert order, tiles are listed expert by expert in decreasing group size, and
        // slot t = c + G*i (CTA c of G, its i-th tile) takes the list's next entry from the front
        // when t is a multiple of 3 and from the back otherwise: front slot t is list position
        // t / 3, back slot t position ntiles - 1 - (t - ceil(t / 3)), one to one for any ntiles.
        // With G not a multiple of 3 each CTA then runs one tile of a long contraction
        // (operand-bound) between two of short ones (master-weight-bound), and at any time a third
        // of the CTAs work on the front.  Otherwise, for even G, slot t takes the front when c + i
        // is even (each CTA alternates; position i * G/2 + c/2 from its end).  The fused SGD lists
        // only the experts that have rows.
        const uint32_t per_e = (uint32_t)p.n_tiles_m * ntn;
        uint32_t l = t32;
        if (p.order != nullptr && gridDim.x % 3u != 0) {
            l = t32 % 3u == 0 ? t32 / 3u : (uint32_t)ntiles - 1 - (t32 - (t32 + 2u) / 3u);
        } else if (p.order != nullptr && (gridDim.x & 1u) == 0) {
            const uint32_t G = gridDim.x, i = t32 / G, c = t32 - i * G;
            const uint32_t fi = i * (G / 2) + c / 2;
            l = ((c + i) & 1) == 0 ? fi : (uint32_t)ntiles - 1 - fi;
        }
        const uint32_t r = l / per_e, rem = l - r * per_e;
        const int e = p.order != nullptr ? __ldg(p.order + r) : (int)r;
        const uint32_t mt = rem / ntn, nt = rem - mt * ntn;
        tl.e = e;
        tl.m0 = (int64_t)mt * BM;
        tl.n0 = (int64_t)nt * BNT;
        tl.b_row = tl.n0;
        const int32_t k0 = __ldg(p.offs + e), k1 = __ldg(p.offs + e + 1);
        tl.k_begin = k0;
        tl.n_stages = (k1 - k0) / Cfg<KIND>::ELEMS;
    }
    return tl;
}

// The largest magnitude of RN(H_128 u / sqrt(128)) over one 128-value row chunk held by one
// thread: butterflies of span 1, 2, ..., 64, (u[i], u[i+h]) <- (u[i] + u[i+h], u[i] - u[i+h]) for i
// with bit h clear, each one binary32 rounding (the order of the return-path codec's transform);
// then, as RN(x * c) is monotone in |x| for c > 0, the largest |u| times c = RN(1/sqrt(128)) is the
// largest rotated magnitude.  u is overwritten.
__device__ __forceinline__ float fwht128_amax(float (&u)[128]) {
#pragma unroll
    for (int h = 1; h < 128; h <<= 1)
#pragma unroll
        for (int i = 0; i < 128; ++i)
            if ((i & h) == 0) {
                const float a = u[i], b = u[i + h];
                u[i] = __fadd_rn(a, b);
                u[i + h] = __fsub_rn(a, b);
            }
    float m = 0.0f;
#pragma unroll
    for (int i = 0; i < 128; ++i) m = fmaxf(m, fabsf(u[i]));
    return __fmul_rn(m, __uint_as_float(0x3DB504F3u));
}

template <int KIND, int EM>
__global__ void __launch_bounds__(THREADS, 1)
    grouped_gemm_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                        const __grid_constant__ CUtensorMap tmW, const __grid_constant__ CUtensorMap tmWb, const Args p) {
    // tmW: the output D (EPI_TMA) or the master weights (EPI_SGD); tmWb: their bf16 copy (EPI_SGD)
    constexpr bool kSgd = is_sgd(EM);
    using Ring = SgdRing<EM>;
    constexpr int NST = EpiCfg<EM>::template NSTK<KIND>;
    constexpr int BNT = EpiCfg<EM>::BNT;
    using L = Layout<KIND, NST, EpiCfg<EM>::template BYTESK<KIND>, BNT>;
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint64_t *bars = reinterpret_cast<uint64_t *>(smem + L::OFF_BAR);
    uint64_t *full = bars, *empty = bars + NST;
    // per accumulator buffer: tmem_full (MMA done) and tmem_empty (epilogue has read it)
    uint64_t *tmem_full = bars + 2 * NST, *tmem_empty = tmem_full + 3, *drain = tmem_full + 6;
    uint64_t *epi_bar = tmem_full + 7;  // fused SGD: Ring::NB per epilogue warp
    uint32_t *tmem_holder = reinterpret_cast<uint32_t *>(smem + L::OFF_MISC);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(smem + L::OFF_MISC + 4);

    const int warp = warp_id(), lane = lane_id();
    // Tiles to run.  The fused SGD skips experts without rows (their weights do not change): with
    // an expert order the list holds only the experts that have rows, order[E] of them.
    const int64_t ntiles = (kSgd && p.order != nullptr)
                               ? (int64_t)__ldg(p.order + p.E) * p.n_tiles_m * p.n_tiles_n
                               : p.num_tiles;
    if (threadIdx.x == 0) {
        for (int s = 0; s < NST; ++s) {
            mbar_init(full + s, 1);
            mbar_init(empty + s, 1);
        }
        for (int i = 0; i < 3; ++i) {
            mbar_init(tmem_full + i, 1);
            mbar_init(tmem_empty + i, EPI_THREADS);
        }
        mbar_init(drain, 1);
        for (int i = 0; i < 8 * Ring::NB; ++i) mbar_init(epi_bar + i, 1);
        *abort_flag = 0;
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    if (warp == 2) {
        asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(tmem_holder)),
                     "r"(TMEM_COLS)
                     : "memory");
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_holder;

    if (warp == 0 && lane == 0) {
        // ---------------------------------------------------------------- producer
        int stage = 0;
        uint32_t phase = 0;
        uint32_t issued_parity[NST];
        bool issued[NST];
        for (int s = 0; s < NST; ++s) issued[s] = false, issued_parity[s] = 0;
        for (int64_t t = blockIdx.x; t < ntiles && !*abort_flag; t += gridDim.x) {
            const Tile tl = decode_tile<KIND, BNT>(p, t, ntiles);
            for (int ks = 0; ks < tl.n_stages; ++ks) {
                if (!mbar_wait(empty + stage, phase ^ 1u, abort_flag)) break;
                uint64_t *fb = full + stage;
                mbar_expect_tx(fb, L::TX);
                const int64_t kel = tl.k_begin + (int64_t)ks * Cfg<KIND>::ELEMS;   // contraction element
                const int xbytes = (int)(KIND == 0 ? kel / 2 : kel);
                tma_load_2d(smem + L::OFF_A + stage * A_TILE, &tmA, fb, xbytes, (int)tl.m0);
                if constexpr (EM == EPI_SWI) {
                    // B rows: the gate slice, then the up slice f rows further on (128-row boxes)
                    tma_load_2d(smem + L::OFF_B + stage * L::B_TILE, &tmB, fb, xbytes, (int)tl.b_row);
                    tma_load_2d(smem + L::OFF_B + stage * L::B_TILE + 128 * BKB, &tmB, fb, xbytes,
                                (int)(tl.b_row + p.swiglu_f));
                } else {
                    tma_load_2d(smem + L::OFF_B + stage * L::B_TILE, &tmB, fb, xbytes, (int)tl.b_row);
                }
                const int64_t atom = kel / Cfg<KIND>::ELEMS_PER_ATOM;
                const uint8_t *sa = p.sfa + ((tl.m0 / BM) * p.sfa_tile_stride + atom) * 512;
                bulk_load(smem + L::OFF_SFA + stage * L::SFA, sa, L::SFA, fb);
                for (int rt = 0; rt < L::RT; ++rt) {
                    // the 128-row tile of B's scales that row tile rt of the stage holds
                    const int64_t brow = (EM == EPI_SWI && rt == 1) ? tl.b_row + p.swiglu_f : tl.b_row + rt * BM;
                    const uint8_t *sb = p.sfb + ((brow / BM) * p.sfb_tile_stride + atom) * 512;
                    bulk_load(smem + L::OFF_SFB + stage * L::SFB + rt * L::SFA, sb, L::SFA, fb);
                }
                issued[stage] = true;
                issued_parity[stage] = phase;
                if (++stage == NST) stage = 0, phase ^= 1u;
            }
        }
        if (*abort_flag) {  // let this CTA's own copies land before the CTA can exit
            for (int s = 0; s < NST; ++s)
                if (issued[s]) {
                    const uint32_t a = smem_u32(full + s);
                    const long long t0 = clock64();
                    while (!mbar_try_wait(a, issued_parity[s]) && clock64() - t0 < kWaitCycles) {
                    }
                }
        }
    } else if (warp == 1 && lane == 0) {
        // ---------------------------------------------------------------- MMA issuer
        int stage = 0;
        uint32_t phase = 0;
        uint32_t acc_ph[3] = {0u, 0u, 0u};
        int acc = 0;  // accumulator buffer of this tile
        const uint32_t a_base = smem_u32(smem + L::OFF_A), b_base = smem_u32(smem + L::OFF_B);
        const uint32_t sfa_base = smem_u32(smem + L::OFF_SFA), sfb_base = smem_u32(smem + L::OFF_SFB);
        for (int64_t t = blockIdx.x; t < ntiles && !*abort_flag; t += gridDim.x) {
            const Tile tl = decode_tile<KIND, BNT>(p, t, ntiles);
            if (kSgd && tl.n_stages == 0) continue;  // an expert without rows: skipped by every role
            if (!mbar_wait(tmem_empty + acc, acc_ph[acc] ^ 1u, abort_flag)) break;
            tc_fence_after();
            const uint32_t tmem_d = tmem + (uint32_t)(acc * BNT);
            if (tl.n_stages == 0) {
                mbar_arrive(tmem_full + acc);
            } else {
                for (int ks = 0; ks < tl.n_stages; ++ks) {
                    if (!mbar_wait(full + stage, phase, abort_flag)) break;
                    tc_fence_after();
                    const uint32_t sf_col = tmem + L::SF_BASE + stage * L::SF_COLS;
                    // scale factors: atom i of A -> columns sf_col + 4i; atom i of B row tile rt ->
                    // sf_col + SF_COLS_A + 4*RT*i + 4rt
#pragma unroll
                    for (int i = 0; i < Cfg<KIND>::ATOMS; ++i) {
                        tc_cp_sf(sf_col + 4 * i, smem_desc(sfa_base + stage * L::SFA + i * 512, 0, 128, 0));
#pragma unroll
                        for (int rt = 0; rt < L::RT; ++rt)
                            tc_cp_sf(sf_col + L::SF_COLS_A + 4 * L::RT * i + 4 * rt,
                                     smem_desc(sfb_base + stage * L::SFB + rt * L::SFA + i * 512, 0, 128, 0));
                    }
                    const uint32_t a_addr = a_base + stage * A_TILE, b_addr = b_base + stage * L::B_TILE;
#pragma unroll
                    for (int k = 0; k < 4; ++k) {
                        const uint64_t ad = smem_desc(a_addr + 32 * k, 16, 1024, 2);
                        const uint64_t bd = smem_desc(b_addr + 32 * k, 16, 1024, 2);
                        uint32_t sfa_t, sfb_t, idesc;
                        if constexpr (KIND == 0) {
                            sfa_t = sf_col + 4 * k;
                            sfb_t = sf_col + L::SF_COLS_A + 4 * L::RT * k;
                            idesc = make_idesc<0, BNT>(0);
                        } else {
                            sfa_t = sf_col;
                            sfb_t = sf_col + L::SF_COLS_A;
                            idesc = make_idesc<1, BNT>((uint32_t)k);
                        }
                        tc_mma<KIND>(tmem_d, ad, bd, idesc, sfa_t, sfb_t, (ks > 0 || k > 0) ? 1u : 0u);
                    }
                    tc_commit(empty + stage);
                    if (++stage == NST) stage = 0, phase ^= 1u;
                }
                tc_commit(tmem_full + acc);
            }
            acc_ph[acc] ^= 1u;
            if (++acc == L::NACC) acc = 0;
        }
        // all of this thread's MMAs and copies complete before tensor memory is freed
        tc_commit(drain);
        const uint32_t a = smem_u32(drain);
        const long long t0 = clock64();
        while (!mbar_try_wait(a, 0) && clock64() - t0 < kWaitCycles) {
        }
    } else if (warp >= 4) {
        // ---------------------------------------------------------------- epilogue
        // warp w reads TMEM lanes 32*(w%4).. (its rows) and half (w-4)/4 of the tile's columns
        const int q = warp & 3;
        const int half = (warp - 4) >> 2;
        uint32_t acc_ph[3] = {0u, 0u, 0u};
        int acc = 0;
        uint32_t sgd_tile = 0, sgd_issued = 0, sgd_done = 0;  // fused SGD: tiles, chunk loads issued / consumed
        uint32_t swb_tile = 0, swb_issued = 0, swb_done = 0;  // SwiGLU backward: the same for its GU chunks
        // SwiGLU backward (lane 0): chunk u of this warp's stream (tile u / 8 of the CTA, columns
        // 16 * (u % 8) of the warp's 128) into buffer u % 2: the gate and the up pieces of GU.  The
        // stores that read that buffer last (chunk u - 2's dg and du) must have read it out first.
        auto swb_issue = [&](uint32_t u, const Tile &tt) {
            const int b = (int)(u & 1u);
            uint8_t *buf = smem + L::OFF_EPI + (warp - 4) * SWB_WARP_BYTES + b * SWB_BUF;
            uint64_t *bar = epi_bar + 2 * (warp - 4) + b;
            bulk_wait_read_all();
            mbar_expect_tx(bar, SWB_BUF);
            const int yy = (int)(tt.m0 + q * 32);
            const int xx = (int)(tt.n0 + half * (BNT / 2) + 16 * (int)(u & 7u));
            tma_load_2d(buf, &tmW, bar, xx, yy);
            tma_load_2d(buf + SWB_BUF / 2, &tmW, bar, (int)(p.swb_f + xx), yy);
        };
        for (int64_t t = blockIdx.x; t < ntiles && !*abort_flag; t += gridDim.x) {
            const Tile tl = decode_tile<KIND, BNT>(p, t, ntiles);
            if (kSgd && tl.n_stages == 0) continue;  // an expert without rows: skipped by every role
            // fused SGD: the CTA's next tile that has rows (its first master-weight chunks are
            // loaded ahead), decoded while the accumulator is still being produced
            int64_t tn = t + gridDim.x;
            Tile tn_l{};
            if constexpr (kSgd || EM == EPI_SWB) {
                for (; tn < ntiles; tn += gridDim.x) {
                    tn_l = decode_tile<KIND, BNT>(p, tn, ntiles);
                    if (tn_l.n_stages > 0) break;
                }
            }
            const bool has_next = tn < ntiles;
            if (!mbar_wait(tmem_full + acc, acc_ph[acc], abort_flag)) break;
            tc_fence_after();
            const bool live = tl.n_stages > 0;
            float alpha = 1.0f;
            if constexpr (KIND == 0) alpha = __fmul_rn(__ldg(p.a_g_dec), __ldg(p.b_g_dec + tl.e));
            const int64_t row = tl.m0 + q * 32 + lane;
            const int64_t dbase = (p.group_k ? (int64_t)tl.e * p.M * p.N : 0) + row * p.N + tl.n0 + half * (BNT / 2);
            const uint32_t tbase = tmem + ((uint32_t)(q * 32) << 16) + (uint32_t)(acc * BNT + half * (BNT / 2));
            if constexpr (kSgd) {
                // W32 <- W32 - lr * dW, bf16 copy, running max |bf16|.  This warp owns rows
                // 32q..32q+31 and columns half*128 .. +127 of the tile, in NCH 16-column chunks.
                // Chunks form one stream over this CTA's tiles: chunk u (tile u / NCH of the CTA,
                // column chunk u % NCH) uses ring buffer u % NB, whose barrier completes for
                // the (u / NB)-th time.  TMA brings the 32x16 binary32 chunk into shared memory
                // (64-byte swizzle: lane l's 16-byte piece j sits at piece j ^ ((l >> 1) & 3) of
                // its 64-byte row), the lane updates its row in place and writes the bf16 row
                // (32-byte swizzle: piece j at j ^ ((l >> 2) & 1)), and TMA stores both.  The load
                // of chunk u + LA is issued before chunk u is processed; it may belong to the
                // CTA's next tile, whose master weights do not depend on that tile's accumulator.
                constexpr int NCH = (BNT / 2) / SGD_CW;
                const int wi = warp - 4;
                constexpr int NB = Ring::NB, LA = Ring::LA;
                uint8_t *wring = smem + L::OFF_EPI + wi * Ring::WARP_BYTES;
                uint8_t *bring = wring + NB * SGD_W_CHUNK;
                uint64_t *eb = epi_bar + NB * wi;
                const int y0 = (int)((int64_t)tl.e * p.M + tl.m0 + q * 32);
                const int x0 = (int)(tl.n0 + half * (BNT / 2));
                int ny0 = 0, nx0 = 0;
                if (has_next) {
                    ny0 = (int)((int64_t)tn_l.e * p.M + tn_l.m0 + q * 32);
                    nx0 = (int)(tn_l.n0 + half * (BNT / 2));
                }
                const uint32_t u0 = sgd_tile * NCH;  // this tile's first chunk in the stream
                // last chunk that may be issued: the end of this tile, or of the next one
                const uint32_t u_end = u0 + (has_next ? 2 * NCH : NCH);
                auto issue = [&](uint32_t u) {  // lane 0
                    const bool nxt = u >= u0 + NCH;
                    const int c = (int)(u % NCH);
                    const int buf = (int)(u % NB);
                    bulk_wait_read_1();  // the store of chunk u - NB, from this buffer, has read it
                    mbar_expect_tx(eb + buf, SGD_W_CHUNK);
                    tma_load_2d(wring + buf * SGD_W_CHUNK, &tmW, eb + buf, (nxt ? nx0 : x0) + SGD_CW * c,
                                nxt ? ny0 : y0);
                };
                while (sgd_issued < u0 + LA && sgd_issued < u_end) {  // the stream's first chunks
                    if (lane == 0) issue(sgd_issued);
                    ++sgd_issued;
                }
                __syncwarp();
                const float lr = p.lr;
                constexpr bool with_bf16 = Ring::BF16;  // else only the amax of the bf16 values
                uint32_t amax2 = 0;
                bool ok = true;
#pragma unroll 1
                for (int c = 0; c < NCH; ++c) {
                    const uint32_t u = u0 + c;
                    if (sgd_issued == u + LA && sgd_issued < u_end) {
                        if (lane == 0) issue(sgd_issued);
                        ++sgd_issued;
                    }
                    __syncwarp();
                    const int buf = (int)(u % NB);
                    ok = __all_sync(0xFFFFFFFFu, mbar_wait(eb + buf, (u / NB) & 1u, abort_flag));
                    if (!ok) break;
                    ++sgd_done;
                    uint32_t r[16];
                    if (live) {
                        tc_ld16(tbase + (uint32_t)(c * SGD_CW), r);
                    } else {
#pragma unroll
                        for (int i = 0; i < 16; ++i) r[i] = 0;
                    }
                    uint8_t *wrow = wring + buf * SGD_W_CHUNK + lane * 64;
                    uint8_t *brow = bring + buf * Ring::B_CHUNK + lane * 32;
                    uint32_t pk[8];
#pragma unroll
                    for (int j = 0; j < 4; ++j) {
                        float4 *slot = reinterpret_cast<float4 *>(wrow + ((j ^ ((lane >> 1) & 3)) << 4));
                        float4 o = *slot;
                        o.x = __fsub_rn(o.x, __fmul_rn(lr, __uint_as_float(r[4 * j])));
                        o.y = __fsub_rn(o.y, __fmul_rn(lr, __uint_as_float(r[4 * j + 1])));
                        o.z = __fsub_rn(o.z, __fmul_rn(lr, __uint_as_float(r[4 * j + 2])));
                        o.w = __fsub_rn(o.w, __fmul_rn(lr, __uint_as_float(r[4 * j + 3])));
                        *slot = o;
                        pk[2 * j] = (uint32_t)f32_to_bf16_bits(o.x) | ((uint32_t)f32_to_bf16_bits(o.y) << 16);
                        pk[2 * j + 1] = (uint32_t)f32_to_bf16_bits(o.z) | ((uint32_t)f32_to_bf16_bits(o.w) << 16);
                        amax2 = __vmaxu2(amax2, pk[2 * j] & 0x7FFF7FFFu);
                        amax2 = __vmaxu2(amax2, pk[2 * j + 1] & 0x7FFF7FFFu);
                    }
                    if constexpr (with_bf16) {
#pragma unroll
                        for (int j = 0; j < 2; ++j)
                            *reinterpret_cast<uint4 *>(brow + ((j ^ ((lane >> 2) & 1)) << 4)) =
                                make_uint4(pk[4 * j], pk[4 * j + 1], pk[4 * j + 2], pk[4 * j + 3]);
                    }
                    fence_async_smem();
                    __syncwarp();
                    if (lane == 0) {
                        if (live) {
                            tma_store_2d(&tmW, wring + buf * SGD_W_CHUNK, x0 + SGD_CW * c, y0);
                            if constexpr (with_bf16)
                                tma_store_2d(&tmWb, bring + buf * Ring::B_CHUNK, x0 + SGD_CW * c, y0);
                        }
                        bulk_commit();  // one group per chunk, empty or not, so group counts match chunks
                    }
                }
                ++sgd_tile;
                uint32_t m = max(amax2 & 0xFFFFu, amax2 >> 16) << 16;
                m = __reduce_max_sync(0xFFFFFFFFu, m);
                if (lane == 0 && m) atomicMax(p.amax + tl.e, m);
                if (!ok) break;
            } else if constexpr (EM == EPI_HMX) {
                // The 8.25-bit return-path codec of the bf16 product, fused: this warp's 32 rows x
                // 128 columns (one 128-chunk per row) go accumulator -> binary32 * alpha -> bf16 ->
                // staging (row = lane), then come back 16 values per lane, 8 lanes per row-chunk,
                // through the Hadamard(128) butterflies and the MXFP8 quantiser (E4M3, one E8M0
                // scale per 32 by the ceiling rule, nearest-even), straight to global memory.
                uint8_t *stg = smem + L::OFF_EPI + (warp - 4) * HMX_WARP_BYTES;
#pragma unroll 1
                for (int c = 0; c < 4; ++c) {
                    uint32_t r[32];
                    if (live) {
                        tc_ld32(tbase + (uint32_t)(c * 32), r);
                    } else {
#pragma unroll
                        for (int i = 0; i < 32; ++i) r[i] = 0;
                    }
                    uint32_t w[16];
#pragma unroll
                    for (int i = 0; i < 16; ++i)
                        w[i] = (uint32_t)f32_to_bf16_bits(__fmul_rn(__uint_as_float(r[2 * i]), alpha)) |
                               ((uint32_t)f32_to_bf16_bits(__fmul_rn(__uint_as_float(r[2 * i + 1]), alpha)) << 16);
                    uint4 *dst = reinterpret_cast<uint4 *>(stg + lane * HMX_PITCH + c * 64);
#pragma unroll
                    for (int j = 0; j < 4; ++j) dst[j] = make_uint4(w[4 * j], w[4 * j + 1], w[4 * j + 2], w[4 * j + 3]);
                }
                // the staged rows are all this warp needs: hand the accumulator back now, so the
                // next tile's MMAs overlap the transform and quantisation below
                tc_fence_before();
                mbar_arrive(tmem_empty + acc);
                __syncwarp();
                const int sub = lane & 7;
                uint8_t *q_out = static_cast<uint8_t *>(p.d);
#pragma unroll 1
                for (int it = 0; it < 8; ++it) {
                    const int rr = 4 * it + (lane >> 3);
                    const uint4 *src = reinterpret_cast<const uint4 *>(stg + rr * HMX_PITCH + sub * 32);
                    const uint4 a0 = src[0], a1 = src[1];
                    const uint32_t hw[8] = {a0.x, a0.y, a0.z, a0.w, a1.x, a1.y, a1.z, a1.w};
                    float u[16];
#pragma unroll
                    for (int i = 0; i < 8; ++i) {
                        u[2 * i] = bf16_lo(hw[i]);
                        u[2 * i + 1] = bf16_hi(hw[i]);
                    }
                    fwht128_sub16(u);
                    float am = 0.0f;
#pragma unroll
                    for (int i = 0; i < 16; ++i) am = fmaxf(am, fabsf(u[i]));
                    am = fmaxf(am, __shfl_xor_sync(0xFFFFFFFFu, am, 1));
                    const int e = mx_scale_exponent(am);
                    const float sc = pow2_neg(e);
                    uint32_t cw[4];
#pragma unroll
                    for (int j = 0; j < 4; ++j)
                        cw[j] = e4m3x4_rn(__fmul_rn(u[4 * j], sc), __fmul_rn(u[4 * j + 1], sc),
                                          __fmul_rn(u[4 * j + 2], sc), __fmul_rn(u[4 * j + 3], sc));
                    const int64_t grow = tl.m0 + q * 32 + rr;
                    const int64_t col = tl.n0 + half * (BNT / 2) + sub * 16;
                    *reinterpret_cast<uint4 *>(q_out + grow * p.N + col) = make_uint4(cw[0], cw[1], cw[2], cw[3]);
                    if ((sub & 1) == 0) p.e8[grow * (p.N / 32) + col / 32] = (uint8_t)(e + 127);
                }
                __syncwarp();  // the staging rows are rewritten by this warp's next tile
            } else if constexpr (EM == EPI_SWB) {
                // dGU = SwiGLU'(GU, dH) for this warp's rows 32q .. 32q + 31 and dH columns
                // x0 .. x0 + 127 (gate columns of GU; the up columns are f further on), 16 columns a
                // chunk: dg = (dh * u) * (s * (1 + g * (1 - s))), du = dh * (g * s), s = 1 / (1 +
                // exp(-g)), each step one binary32 rounding, then bf16, as moe4_swiglu_backward
                // computes them from dH.  The slab of dH goes to registers and the accumulator is
                // handed back first; chunk u + 1's GU pieces load while chunk u is processed (the
                // last chunk's successor is the next tile's first).
                const int wi = warp - 4;
                uint8_t *ringw = smem + L::OFF_EPI + wi * SWB_WARP_BYTES;
                const int y0 = (int)(tl.m0 + q * 32);
                const int x0 = (int)(tl.n0 + half * (BNT / 2));
                const uint32_t u0 = swb_tile * 8;
                if (swb_issued == u0) {  // not loaded ahead (the CTA's first tile)
                    if (lane == 0) swb_issue(u0, tl);
                    ++swb_issued;
                }
                uint32_t accr[128];
                if (live) {
#pragma unroll
                    for (int c = 0; c < 4; ++c) tc_ld32_nw(tbase + (uint32_t)(c * 32), accr + 32 * c);
                    tc_wait_ld();
                } else {
#pragma unroll
                    for (int i = 0; i < 128; ++i) accr[i] = 0;
                }
                tc_fence_before();
                mbar_arrive(tmem_empty + acc);
                bool ok = true;
#pragma unroll
                for (int c = 0; c < 8; ++c) {
                    const uint32_t u = u0 + c;
                    if (c + 1 < 8) {
                        if (lane == 0) swb_issue(u + 1, tl);
                        ++swb_issued;
                    } else if (has_next) {
                        if (lane == 0) swb_issue(u + 1, tn_l);
                        ++swb_issued;
                    }
                    __syncwarp();
                    const int b = (int)(u & 1u);
                    ok = __all_sync(0xFFFFFFFFu, mbar_wait(epi_bar + 2 * wi + b, (u >> 1) & 1u, abort_flag));
                    if (!ok) break;
                    ++swb_done;
                    uint8_t *gbuf = ringw + b * SWB_BUF;
                    uint8_t *ubuf = gbuf + SWB_BUF / 2;
                    float gv[16], uv[16];
#pragma unroll
                    for (int j = 0; j < 4; ++j) {
                        const int piece = (j ^ ((lane >> 1) & 3)) << 4;
                        const float4 a4 = *reinterpret_cast<const float4 *>(gbuf + lane * 64 + piece);
                        const float4 b4 = *reinterpret_cast<const float4 *>(ubuf + lane * 64 + piece);
                        gv[4 * j] = a4.x, gv[4 * j + 1] = a4.y, gv[4 * j + 2] = a4.z, gv[4 * j + 3] = a4.w;
                        uv[4 * j] = b4.x, uv[4 * j + 1] = b4.y, uv[4 * j + 2] = b4.z, uv[4 * j + 3] = b4.w;
                    }
                    __syncwarp();  // every lane holds its gate row before dg is written over the chunk
                    uint32_t og[8], ou[8];
#pragma unroll
                    for (int i = 0; i < 8; ++i) og[i] = ou[i] = 0u;
#pragma unroll
                    for (int i = 0; i < 16; ++i) {
                        const float dh = __uint_as_float(accr[16 * c + i]);
                        const float sg = __frcp_rn(__fadd_rn(1.0f, expf(-gv[i])));
                        const float silu = __fmul_rn(gv[i], sg);
                        const float dsilu = __fmul_rn(sg, __fadd_rn(1.0f, __fmul_rn(gv[i], __fsub_rn(1.0f, sg))));
                        og[i >> 1] |= (uint32_t)f32_to_bf16_bits(__fmul_rn(__fmul_rn(dh, uv[i]), dsilu)) << (16 * (i & 1));
                        ou[i >> 1] |= (uint32_t)f32_to_bf16_bits(__fmul_rn(dh, silu)) << (16 * (i & 1));
                    }
                    // 32-byte bf16 rows, 32-byte swizzle: piece j of row l at j ^ ((l >> 2) & 1)
#pragma unroll
                    for (int j = 0; j < 2; ++j) {
                        const int piece = (j ^ ((lane >> 2) & 1)) << 4;
                        *reinterpret_cast<uint4 *>(gbuf + lane * 32 + piece) =
                            make_uint4(og[4 * j], og[4 * j + 1], og[4 * j + 2], og[4 * j + 3]);
                        *reinterpret_cast<uint4 *>(gbuf + 1024 + lane * 32 + piece) =
                            make_uint4(ou[4 * j], ou[4 * j + 1], ou[4 * j + 2], ou[4 * j + 3]);
                    }
                    fence_async_smem();
                    __syncwarp();
                    if (lane == 0) {
                        tma_store_2d(&tmWb, gbuf, x0 + 16 * c, y0);
                        tma_store_2d(&tmWb, gbuf + 1024, (int)(p.swb_f + x0 + 16 * c), y0);
                        bulk_commit();
                    }
                }
                ++swb_tile;
                if (!ok) break;
            } else if constexpr (EM == EPI_SWI) {
                // This warp: rows 32q .. 32q + 31, gate columns 64 * half .. + 63 of the tile
                // (accumulator columns 64 * half ..) and the same columns of up (accumulator
                // columns 128 + 64 * half ..).  Both slabs go to registers and the accumulator is
                // handed back; then six 32-column chunks pass through the staging tile to TMA:
                // GU [M, 2f] binary32 (gate at column n0 + 64 * half, up f columns further on) and
                // h = RN_bf16(silu(g) * u), silu(g) = g / (1 + exp(-g)), each step one binary32
                // rounding, as moe4_swiglu computes it from the same GU values.
                uint8_t *stage = smem + L::OFF_EPI + (warp - 4) * EPI_W_TILE<KIND>;
                const int y0 = (int)(tl.m0 + q * 32);
                const int xg = (int)(tl.n0 + half * 64);
                const uint32_t tg = tmem + ((uint32_t)(q * 32) << 16) + (uint32_t)(acc * BNT + half * 64);
                uint32_t accr[128];  // gate 0 .. 63, up 64 .. 127
                if (live) {
                    tc_ld32_nw(tg, accr);
                    tc_ld32_nw(tg + 32, accr + 32);
                    tc_ld32_nw(tg + 128, accr + 64);
                    tc_ld32_nw(tg + 160, accr + 96);
                    tc_wait_ld();
                } else {
#pragma unroll
                    for (int i = 0; i < 128; ++i) accr[i] = 0;
                }
                tc_fence_before();
                mbar_arrive(tmem_empty + acc);
                uint32_t best = 0;  // two packed bf16 magnitudes of h
#pragma unroll
                for (int c = 0; c < 6; ++c) {  // gate 0, gate 1, up 0, up 1, h 0, h 1
                    if (lane == 0) bulk_wait_read_all();  // the previous store has read the tile out
                    __syncwarp();
                    if (c < 4) {
                        const int off = (c < 2 ? 0 : 64) + (c & 1) * 32;
                        uint8_t *row = stage + lane * 128;  // 32 binary32, 128-byte swizzle
#pragma unroll
                        for (int j = 0; j < 8; ++j) {
                            float o[4];
#pragma unroll
                            for (int i = 0; i < 4; ++i) o[i] = __fmul_rn(__uint_as_float(accr[off + 4 * j + i]), alpha);
                            *reinterpret_cast<float4 *>(row + ((j ^ (lane & 7)) << 4)) = make_float4(o[0], o[1], o[2], o[3]);
                        }
                    } else {
                        const int cc = (c - 4) * 32;
                        uint8_t *row = stage + lane * 64;  // 32 bf16, 64-byte swizzle
#pragma unroll
                        for (int j = 0; j < 4; ++j) {
                            uint32_t w[4];
#pragma unroll
                            for (int i = 0; i < 4; ++i) {
                                uint32_t hb[2];
#pragma unroll
                                for (int e2 = 0; e2 < 2; ++e2) {
                                    const int col = cc + 8 * j + 2 * i + e2;
                                    const float gv = __fmul_rn(__uint_as_float(accr[col]), alpha);
                                    const float uv = __fmul_rn(__uint_as_float(accr[64 + col]), alpha);
                                    const float silu = __fdiv_rn(gv, __fadd_rn(1.0f, expf(-gv)));
                                    hb[e2] = (uint32_t)f32_to_bf16_bits(__fmul_rn(silu, uv));
                                }
                                w[i] = hb[0] | (hb[1] << 16);
                                best = __vmaxu2(best, w[i] & 0x7FFF7FFFu);
                            }
                            *reinterpret_cast<uint4 *>(row + ((j ^ ((lane >> 1) & 3)) << 4)) =
                                make_uint4(w[0], w[1], w[2], w[3]);
                        }
                    }
                    fence_async_smem();
                    __syncwarp();
                    if (lane == 0) {
                        if (c < 4)
                            tma_store_2d(&tmW, stage, (c < 2 ? xg : (int)(p.swiglu_f + xg)) + (c & 1) * 32, y0);
                        else
                            tma_store_2d(&tmWb, stage, xg + (c - 4) * 32, y0);
                        bulk_commit();
                    }
                }
                uint32_t mag = max(best & 0xFFFFu, best >> 16) << 16;
                mag = __reduce_max_sync(0xFFFFFFFFu, mag);
                if (lane == 0 && mag) atomicMax(p.h_amax, mag);
            } else if constexpr (EM == EPI_TMA) {
                // each CW-column chunk: registers -> swizzled 32 x CW staging tile -> TMA bulk store.
                // A staged row is CW * 4 (binary32) or CW * 2 (bf16) bytes with the swizzle of that
                // width: with P 16-byte pieces per row, piece j of row l sits at
                // j ^ ((l >> (3 - log2 P)) & (P - 1))
                constexpr int CW = TMA_CW<KIND>;
                constexpr int PF = CW / 4, PB = CW / 8;            // pieces per binary32 / bf16 row
                constexpr int SF = PF == 8 ? 0 : (PF == 4 ? 1 : 2);  // 3 - log2(PF)
                constexpr int SB = PB == 8 ? 0 : (PB == 4 ? 1 : 2);
                uint8_t *stage = smem + L::OFF_EPI + (warp - 4) * EPI_W_TILE<KIND>;
                const int y0 = (int)((p.group_k ? (int64_t)tl.e * p.M : 0) + tl.m0 + q * 32);
                const int x0 = (int)(tl.n0 + half * (BNT / 2));
                // the warp's whole slab (32 rows x BNT/2 columns) goes to registers first and the
                // accumulator is handed back at once, so the next tile's MMAs run while this tile
                // is converted and stored
                constexpr int NCOL = BNT / 2;
                uint32_t accr[NCOL];
                if (live) {
#pragma unroll
                    for (int c = 0; c < NCOL / 32; ++c) tc_ld32_nw(tbase + (uint32_t)(c * 32), accr + 32 * c);
                    tc_wait_ld();
                } else {
#pragma unroll
                    for (int i = 0; i < NCOL; ++i) accr[i] = 0;
                }
                tc_fence_before();
                mbar_arrive(tmem_empty + acc);
#pragma unroll
                for (int c = 0; c < NCOL / CW; ++c) {
                    float v[CW];
#pragma unroll
                    for (int i = 0; i < CW; ++i)
                        v[i] = KIND == 0 ? __fmul_rn(__uint_as_float(accr[c * CW + i]), alpha)
                                         : __uint_as_float(accr[c * CW + i]);
                    if (lane == 0) bulk_wait_read_all();  // the previous store has read the tile out
                    __syncwarp();
                    if (p.mode == BF16) {
                        uint8_t *row = stage + lane * (CW * 2);
#pragma unroll
                        for (int j = 0; j < PB; ++j) {
                            uint32_t w[4];
#pragma unroll
                            for (int i = 0; i < 4; ++i)
                                w[i] = (uint32_t)f32_to_bf16_bits(v[8 * j + 2 * i]) |
                                       ((uint32_t)f32_to_bf16_bits(v[8 * j + 2 * i + 1]) << 16);
                            *reinterpret_cast<uint4 *>(row + ((j ^ ((lane >> SB) & (PB - 1))) << 4)) =
                                make_uint4(w[0], w[1], w[2], w[3]);
                        }
                    } else {
                        uint8_t *row = stage + lane * (CW * 4);
#pragma unroll
                        for (int j = 0; j < PF; ++j)
                            *reinterpret_cast<float4 *>(row + ((j ^ ((lane >> SF) & (PF - 1))) << 4)) =
                                make_float4(v[4 * j], v[4 * j + 1], v[4 * j + 2], v[4 * j + 3]);
                    }
                    fence_async_smem();
                    __syncwarp();
                    if (lane == 0) {
                        tma_store_2d(&tmW, stage, x0 + CW * c, y0);
                        bulk_commit();
                    }
                }
                if constexpr (KIND == 0 && NCOL == 128) {
                    // the return path's amax: this lane's row chunk (columns x0 .. x0+127, one whole
                    // Hadamard chunk) as the bf16 values just stored, rotated in registers
                    if (p.had_amax != nullptr) {
                        float u[128];
#pragma unroll
                        for (int i = 0; i < 128; ++i)
                            u[i] = __uint_as_float((uint32_t)f32_to_bf16_bits(
                                                       __fmul_rn(__uint_as_float(accr[i]), alpha)) << 16);
                        uint32_t m = __float_as_uint(fwht128_amax(u));
                        m = __reduce_max_sync(0xFFFFFFFFu, m);
                        if (lane == 0 && m) atomicMax(p.had_amax, m);
                    }
                }
            } else {
                for (int c = 0; c < BNT / 64; ++c) {
                    uint32_t r[32];
                    if (live) {
                        tc_ld32(tbase + (uint32_t)(c * 32), r);
                    } else {
#pragma unroll
                        for (int i = 0; i < 32; ++i) r[i] = 0;
                    }
                    float v[32];
#pragma unroll
                    for (int i = 0; i < 32; ++i)
                        v[i] = KIND == 0 ? __fmul_rn(__uint_as_float(r[i]), alpha) : __uint_as_float(r[i]);
                    if (p.mode == BF16) {
                        uint4 *dst = reinterpret_cast<uint4 *>(static_cast<uint16_t *>(p.d) + dbase + c * 32);
#pragma unroll
                        for (int j = 0; j < 4; ++j) {
                            uint32_t w[4];
#pragma unroll
                            for (int i = 0; i < 4; ++i)
                                w[i] = (uint32_t)f32_to_bf16_bits(v[8 * j + 2 * i]) |
                                       ((uint32_t)f32_to_bf16_bits(v[8 * j + 2 * i + 1]) << 16);
                            dst[j] = make_uint4(w[0], w[1], w[2], w[3]);
                        }
                    } else if (p.mode == ACC_F32) {
                        if (!live) continue;
                        float4 *dst = reinterpret_cast<float4 *>(static_cast<float *>(p.d) + dbase + c * 32);
#pragma unroll
                        for (int j = 0; j < 8; ++j) {
                            float4 o = dst[j];
                            o.x = __fadd_rn(o.x, v[4 * j]);
                            o.y = __fadd_rn(o.y, v[4 * j + 1]);
                            o.z = __fadd_rn(o.z, v[4 * j + 2]);
                            o.w = __fadd_rn(o.w, v[4 * j + 3]);
                            dst[j] = o;
                        }
                    } else {
                        float4 *dst = reinterpret_cast<float4 *>(static_cast<float *>(p.d) + dbase + c * 32);
#pragma unroll
                        for (int j = 0; j < 8; ++j) dst[j] = make_float4(v[4 * j], v[4 * j + 1], v[4 * j + 2], v[4 * j + 3]);
                    }
                }
            }
            if constexpr (EM != EPI_HMX && EM != EPI_TMA && EM != EPI_SWI && EM != EPI_SWB) {  // those hand it back early
                tc_fence_before();
                mbar_arrive(tmem_empty + acc);
            }
            acc_ph[acc] ^= 1u;
            if (++acc == L::NACC) acc = 0;
        }
        if constexpr (EM == EPI_SWB) {
            // GU chunk loads the loop did not consume (it stopped early): let them land
            if (lane == 0) {
                for (uint32_t u = swb_done; u < swb_issued; ++u) {
                    const uint32_t aa = smem_u32(epi_bar + 2 * (warp - 4) + (u & 1u));
                    const long long t0 = clock64();
                    while (!mbar_try_wait(aa, (u >> 1) & 1u) && clock64() - t0 < kWaitCycles) {
                    }
                }
            }
        }
        if constexpr (kSgd) {
            // master-weight loads the loop did not consume (it stopped early): let them land
            if (lane == 0) {
                for (uint32_t u = sgd_done; u < sgd_issued; ++u) {
                    const uint32_t aa = smem_u32(epi_bar + Ring::NB * (warp - 4) + u % Ring::NB);
                    const long long t0 = clock64();
                    while (!mbar_try_wait(aa, (u / Ring::NB) & 1u) && clock64() - t0 < kWaitCycles) {
                    }
                }
            }
        }
        if constexpr (EM != EPI_REG) {
            if (lane == 0) bulk_wait_all();  // this warp's stores are complete before the CTA exits
        }
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp == 2) {
        asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(TMEM_COLS) : "memory");
    }
}

// ------------------------------------------------------------------ host side
typedef CUresult (*EncodeTiledFn)(CUtensorMap *, CUtensorMapDataType, cuuint32_t, void *, const cuuint64_t *,
                                  const cuuint64_t *, const cuuint32_t *, const cuuint32_t *, CUtensorMapInterleave,
                                  CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

static EncodeTiledFn encode_fn() {
    static EncodeTiledFn fn = nullptr;
    if (!fn) {
        void *ptr = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<EncodeTiledFn>(ptr);
    }
    return fn;
}

// 2-D tensor [rows, inner] of `elem`-byte elements; box of box_rows x box_inner elements.
static bool make_map_t(CUtensorMap *m, CUtensorMapDataType type, int elem, const void *base, int64_t inner,
                       int64_t rows, int box_inner, int box_rows, CUtensorMapSwizzle swz) {
    EncodeTiledFn enc = encode_fn();
    if (!enc) return false;
    cuuint64_t dims[2] = {(cuuint64_t)inner, (cuuint64_t)rows};
    cuuint64_t strides[1] = {(cuuint64_t)(inner * elem)};
    cuuint32_t box[2] = {(cuuint32_t)box_inner, (cuuint32_t)box_rows};
    cuuint32_t estr[2] = {1, 1};
    return enc(m, type, 2, const_cast<void *>(base), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, swz,
               CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// Operand tile: [rows, inner_bytes] bytes, box box_rows x 128 bytes, 128-byte swizzle.
static bool make_map(CUtensorMap *m, const void *base, int64_t inner_bytes, int64_t rows, int box_rows) {
    return make_map_t(m, CU_TENSOR_MAP_DATA_TYPE_UINT8, 1, base, inner_bytes, rows, BKB, box_rows,
                      CU_TENSOR_MAP_SWIZZLE_128B);
}

template <int KIND, int EM>
static int launch(const CUtensorMap &ta, const CUtensorMap &tb, const CUtensorMap &tw, const CUtensorMap &twb,
                  const Args &a, cudaStream_t st) {
    using L = Layout<KIND, EpiCfg<EM>::template NSTK<KIND>, EpiCfg<EM>::template BYTESK<KIND>, EpiCfg<EM>::BNT>;
    // the dynamic shared-memory limit is an attribute of the kernel in the current context: set
    // on every call (a host-side call), so it also holds after the context has been torn down
    // and created again (cudaDeviceReset), which forgets it
    if (cudaFuncSetAttribute(grouped_gemm_kernel<KIND, EM>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             L::SMEM) != cudaSuccess)
        return MOE4_ERR_CUDA;
    if (a.num_tiles == 0) return MOE4_OK;
    const int64_t grid = a.num_tiles < num_sms() ? a.num_tiles : num_sms();
    grouped_gemm_kernel<KIND, EM><<<(unsigned)grid, THREADS, L::SMEM, st>>>(ta, tb, tw, twb, a);
    return launch_status();
}

// The output D as [rows, N] for the TMA-store epilogue: cw-column x 32-row boxes (cw 32 or 16) with
// the swizzle of the staged row's width.
static CUtensorMapSwizzle swizzle_for(int row_bytes) {
    return row_bytes == 128 ? CU_TENSOR_MAP_SWIZZLE_128B
                            : (row_bytes == 64 ? CU_TENSOR_MAP_SWIZZLE_64B : CU_TENSOR_MAP_SWIZZLE_32B);
}
static bool make_out_map(CUtensorMap *m, void *d, bool bf16, int64_t rows, int64_t N, int cw) {
    return bf16 ? make_map_t(m, CU_TENSOR_MAP_DATA_TYPE_UINT16, 2, d, N, rows, cw, 32, swizzle_for(cw * 2))
                : make_map_t(m, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 4, d, N, rows, cw, 32, swizzle_for(cw * 4));
}

// A wait that nothing completes, through the GEMMs' bounded-wait path: phase 0 of a fresh
// mbarrier with no arrivals.  It gives up after `limit` cycles and records the timeout.
__global__ void wait_selftest_kernel(long long limit) {
    __shared__ __align__(8) uint64_t bar;
    __shared__ int abort_flag;
    if (threadIdx.x == 0) {
        mbar_init(&bar, 1);
        abort_flag = 0;
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    __syncthreads();
    if (threadIdx.x == 0) mbar_wait(&bar, 0u, &abort_flag, limit);
}

// Throughput of the tensor pipe on one CTA per SM: one stage of operands stays in shared memory
// (128 x 128-byte A, 256 x 128-byte B with their scale factors), the scale factors are copied into
// tensor memory once, and the issuing thread runs `iters` rounds of the GEMM's four block-scaled
// MMAs (128 x 256 x 256 FP4 or 128 x 256 x 128 FP8 per round) into one binary32 accumulator,
// then commits once and waits (bounded).  No operand traffic: the rate is the pipe's own.  With
// kCopySf every round first copies its scale factors into tensor memory again, into one of four
// column sets in turn, as the GEMM does for each operand stage.
template <int KIND, bool kCopySf>
__global__ void __launch_bounds__(128, 1) mma_peak_kernel(int64_t iters, uint32_t *sink) {
    constexpr int SFA = Cfg<KIND>::ATOMS * 512, SFB = 2 * SFA;
    constexpr int OFF_B = A_TILE, OFF_SFA = OFF_B + BN * BKB, OFF_SFB = OFF_SFA + SFA, OFF_BAR = OFF_SFB + SFB;
    constexpr int SF_COLS_A = Cfg<KIND>::ATOMS * 4;
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint64_t *done = reinterpret_cast<uint64_t *>(smem + OFF_BAR);
    uint32_t *tmem_holder = reinterpret_cast<uint32_t *>(smem + OFF_BAR + 8);
    int *abort_flag = reinterpret_cast<int *>(smem + OFF_BAR + 12);
    // operands: a hash pattern of valid FP4 / E4M3 codes (no NaN), scales 1.0
    for (int i = threadIdx.x; i < OFF_SFA / 4; i += blockDim.x) {
        uint32_t h = (uint32_t)i * 2654435761u;
        h ^= h >> 15;
        reinterpret_cast<uint32_t *>(smem)[i] = KIND == 0 ? h : (h & 0x77777777u);
    }
    const uint8_t one = KIND == 0 ? 0x38 : 127;  // E4M3 1.0, E8M0 2^0
    for (int i = threadIdx.x; i < SFA + SFB; i += blockDim.x) smem[OFF_SFA + i] = one;
    if (threadIdx.x == 0) {
        mbar_init(done, 1);
        *abort_flag = 0;
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    fence_async_smem();
    if (warp_id() == 0) {
        asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(tmem_holder)),
                     "r"(TMEM_COLS)
                     : "memory");
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_holder;
    if (threadIdx.x == 0) {
        constexpr uint32_t SF_SET = 3 * SF_COLS_A;  // A and two row tiles of B
        const uint32_t sfa_base = smem_u32(smem + OFF_SFA), sfb_base = smem_u32(smem + OFF_SFB);
        auto copy_sf = [&](uint32_t sf_col) {
#pragma unroll
            for (int i = 0; i < Cfg<KIND>::ATOMS; ++i) {
                tc_cp_sf(sf_col + 4 * i, smem_desc(sfa_base + i * 512, 0, 128, 0));
#pragma unroll
                for (int rt = 0; rt < 2; ++rt)
                    tc_cp_sf(sf_col + SF_COLS_A + 8 * i + 4 * rt, smem_desc(sfb_base + rt * SFA + i * 512, 0, 128, 0));
            }
        };
        copy_sf(tmem + BN);
        const uint32_t a_addr = smem_u32(smem), b_addr = smem_u32(smem + OFF_B);
#pragma unroll 1
        for (int64_t it = 0; it < iters; ++it) {
            uint32_t sf_col = tmem + BN;
            if constexpr (kCopySf) {
                sf_col += (uint32_t)(it & 3) * SF_SET;
                copy_sf(sf_col);
            }
#pragma unroll
            for (int k = 0; k < 4; ++k) {
                const uint64_t ad = smem_desc(a_addr + 32 * k, 16, 1024, 2);
                const uint64_t bd = smem_desc(b_addr + 32 * k, 16, 1024, 2);
                if constexpr (KIND == 0)
                    tc_mma<0>(tmem, ad, bd, make_idesc<0, BN>(0), sf_col + 4 * k, sf_col + SF_COLS_A + 8 * k,
                              (it > 0 || k > 0) ? 1u : 0u);
                else
                    tc_mma<1>(tmem, ad, bd, make_idesc<1, BN>((uint32_t)k), sf_col, sf_col + SF_COLS_A,
                              (it > 0 || k > 0) ? 1u : 0u);
            }
        }
        tc_commit(done);
        mbar_wait(done, 0u, abort_flag);
    }
    __syncthreads();
    tc_fence_after();
    uint32_t r[32];
    tc_ld32(tmem + ((uint32_t)(warp_id() * 32) << 16), r);  // keeps the accumulator live
    if (lane_id() == 0 && r[0] == 0x7FC00001u) sink[blockIdx.x] = r[1];
    tc_fence_before();
    __syncthreads();
    if (warp_id() == 0)
        asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(TMEM_COLS) : "memory");
}

}  // namespace gemm
}  // namespace moe4

using namespace moe4;
using namespace moe4::gemm;

extern "C" int moe4_get_status(void *stream) {
    if (cudaStreamSynchronize(as_stream(stream)) != cudaSuccess) return MOE4_ERR_CUDA;
    unsigned int v = 0, zero = 0;
    if (cudaMemcpyFromSymbol(&v, g_status, sizeof(v)) != cudaSuccess) return MOE4_ERR_CUDA;
    if (v && cudaMemcpyToSymbol(g_status, &zero, sizeof(zero)) != cudaSuccess) return MOE4_ERR_CUDA;
    return v ? MOE4_ERR_TIMEOUT : MOE4_OK;
}

// Before the fused SGD: amax_out[e] = 0 for every expert that has rows (the others are skipped
// and keep theirs), and, when `order` is given (E < 4096), the experts that have rows by
// decreasing group size (ties by index) in order[0 .. L) with L = order[E].
__global__ void __launch_bounds__(1024) sgd_prep_kernel(const int32_t *__restrict__ offs, int E,
                                                        int32_t *__restrict__ order, unsigned int *__restrict__ amax) {
    __shared__ int32_t sz[4096];
    __shared__ int live;
    if (threadIdx.x == 0) live = 0;
    __syncthreads();
    for (int e = threadIdx.x; e < E; e += blockDim.x) {
        const int32_t n = __ldg(offs + e + 1) - __ldg(offs + e);
        if (n > 0) {
            amax[e] = 0u;
            atomicAdd(&live, 1);
        }
        if (order != nullptr) sz[e] = n;
    }
    __syncthreads();
    if (order == nullptr) return;
    for (int e = threadIdx.x; e < E; e += blockDim.x) {
        const int ke = sz[e];
        if (ke == 0) continue;
        int rank = 0;
        for (int j = 0; j < E; ++j) rank += (sz[j] > ke) || (sz[j] == ke && j < e);
        order[rank] = e;
    }
    if (threadIdx.x == 0) order[E] = live;
}

// Whether ws holds the tensor-core copies of both operands' scale factors.
static bool scales_ws_ok(int64_t a_rows, int64_t b_rows, int64_t K, int blk, const void *ws, size_t ws_bytes) {
    const size_t na = (size_t)(a_rows * (K / blk)), nb = (size_t)(b_rows * (K / blk));
    const size_t need = (na + 255) / 256 * 256 + (nb + 255) / 256 * 256;
    return ws && ws_bytes >= need && aligned16(ws);
}

// Canonical scales -> tensor-core layout into ws when the caller did not pass that layout.
static int stage_scales(const uint8_t *a_sf, int64_t a_rows, const uint8_t *b_sf, int64_t b_rows, int64_t K, int blk,
                        uint32_t flags, void *ws, size_t ws_bytes, const uint8_t **sfa, const uint8_t **sfb,
                        cudaStream_t st) {
    if (flags & MOE4_SF_MMA_LAYOUT) {
        *sfa = a_sf;
        *sfb = b_sf;
        return MOE4_OK;
    }
    if (!scales_ws_ok(a_rows, b_rows, K, blk, ws, ws_bytes)) return MOE4_ERR_WORKSPACE;
    const size_t na = (size_t)(a_rows * (K / blk));
    uint8_t *wa = static_cast<uint8_t *>(ws);
    uint8_t *wb = wa + (na + 255) / 256 * 256;
    int rc = moe4_sf_to_mma_layout(a_sf, 1, a_rows, K / blk, wa, st);
    if (rc == MOE4_OK) rc = moe4_sf_to_mma_layout(b_sf, 1, b_rows, K / blk, wb, st);
    *sfa = wa;
    *sfb = wb;
    return rc;
}

extern "C" int grouped_expert_gemm_nvfp4(const uint8_t *a_codes, const uint8_t *a_sf, const float *a_g_dec,
                                         const uint8_t *b_codes, const uint8_t *b_sf, const float *b_g_dec,
                                         const int32_t *group_offs, int64_t E, int64_t rows_total, int64_t N,
                                         int64_t K, void *d, uint32_t flags, void *ws, size_t ws_bytes,
                                         void *stream) {
    MOE4_CHECK_ARG(E >= 1 && rows_total >= 0 && rows_total % BM == 0 && N > 0 && N % BN == 0 && K > 0 &&
                   K % 256 == 0);
    MOE4_CHECK_ARG(a_codes && a_sf && a_g_dec && b_codes && b_sf && b_g_dec && group_offs && d);
    MOE4_CHECK_ARG(aligned16(a_codes) && aligned16(b_codes) && aligned16(a_sf) && aligned16(b_sf) && aligned16(d));
    MOE4_CHECK_ARG((flags & ~(MOE4_OUT_F32 | MOE4_OUT_BF16 | MOE4_SF_MMA_LAYOUT)) == 0);
    const bool bf16 = (flags & MOE4_OUT_BF16) != 0;
    MOE4_CHECK_ARG(bf16 != ((flags & MOE4_OUT_F32) != 0));
    MOE4_CHECK_ARG(rows_total < (int64_t(1) << 31) && E * N < (int64_t(1) << 31));
    if (rows_total == 0) return MOE4_OK;
    cudaStream_t st = as_stream(stream);
    const uint8_t *sfa, *sfb;
    int rc = stage_scales(a_sf, rows_total, b_sf, E * N, K, 16, flags, ws, ws_bytes, &sfa, &sfb, st);
    if (rc != MOE4_OK) return rc;
    CUtensorMap ta, tb;
    if (!make_map(&ta, a_codes, K / 2, rows_total, BM) || !make_map(&tb, b_codes, K / 2, E * N, BN))
        return MOE4_ERR_CUDA;
    Args a{};
    a.sfa = sfa;
    a.sfb = sfb;
    a.a_g_dec = a_g_dec;
    a.b_g_dec = b_g_dec;
    a.offs = group_offs;
    a.E = (int)E;
    a.group_k = 0;
    a.M = rows_total;
    a.N = N;
    a.K = K;
    a.d = d;
    a.mode = bf16 ? BF16 : F32;
    a.n_tiles_n = (int)(N / BN);
    a.n_tiles_m = (int)(rows_total / BM);
    a.num_tiles = (int64_t)a.n_tiles_m * a.n_tiles_n;
    a.sfa_tile_stride = K / 64;
    a.sfb_tile_stride = K / 64;
    CUtensorMap td;
    if (!make_out_map(&td, d, bf16, rows_total, N, TMA_CW<0>)) return MOE4_ERR_CUDA;
    return launch<0, EPI_TMA>(ta, tb, td, td, a, st);
}

extern "C" int grouped_expert_gemm_nvfp4_hadamard_amax(const uint8_t *a_codes, const uint8_t *a_sf,
                                                       const float *a_g_dec, const uint8_t *b_codes,
                                                       const uint8_t *b_sf, const float *b_g_dec,
                                                       const int32_t *group_offs, int64_t E, int64_t rows_total,
                                                       int64_t N, int64_t K, uint16_t *d, float *amax_out,
                                                       uint32_t flags, void *ws, size_t ws_bytes, void *stream) {
    MOE4_CHECK_ARG(E >= 1 && rows_total >= 0 && rows_total % BM == 0 && N > 0 && N % BN == 0 && K > 0 &&
                   K % 256 == 0);
    MOE4_CHECK_ARG(a_codes && a_sf && a_g_dec && b_codes && b_sf && b_g_dec && group_offs && d && amax_out);
    MOE4_CHECK_ARG(aligned16(a_codes) && aligned16(b_codes) && aligned16(a_sf) && aligned16(b_sf) && aligned16(d) &&
                   aligned4(amax_out));
    MOE4_CHECK_ARG((flags & ~MOE4_SF_MMA_LAYOUT) == 0);
    MOE4_CHECK_ARG(rows_total < (int64_t(1) << 31) && E * N < (int64_t(1) << 31));
    // a missing workspace is reported before anything is enqueued
    if (rows_total > 0 && !(flags & MOE4_SF_MMA_LAYOUT) && !scales_ws_ok(rows_total, E * N, K, 16, ws, ws_bytes))
        return MOE4_ERR_WORKSPACE;
    cudaStream_t st = as_stream(stream);
    if (cudaMemsetAsync(amax_out, 0, sizeof(float), st) != cudaSuccess) return MOE4_ERR_CUDA;
    if (rows_total == 0) return MOE4_OK;
    const uint8_t *sfa, *sfb;
    int rc = stage_scales(a_sf, rows_total, b_sf, E * N, K, 16, flags, ws, ws_bytes, &sfa, &sfb, st);
    if (rc != MOE4_OK) return rc;
    CUtensorMap ta, tb;
    if (!make_map(&ta, a_codes, K / 2, rows_total, BM) || !make_map(&tb, b_codes, K / 2, E * N, BN))
        return MOE4_ERR_CUDA;
    Args a{};
    a.sfa = sfa;
    a.sfb = sfb;
    a.a_g_dec = a_g_dec;
    a.b_g_dec = b_g_dec;
    a.offs = group_offs;
    a.E = (int)E;
    a.group_k = 0;
    a.M = rows_total;
    a.N = N;
    a.K = K;
    a.d = d;
    a.mode = BF16;
    a.had_amax = reinterpret_cast<unsigned int *>(amax_out);
    a.n_tiles_n = (int)(N / BN);
    a.n_tiles_m = (int)(rows_total / BM);
    a.num_tiles = (int64_t)a.n_tiles_m * a.n_tiles_n;
    a.sfa_tile_stride = K / 64;
    a.sfb_tile_stride = K / 64;
    CUtensorMap td;
    if (!make_out_map(&td, d, true, rows_total, N, TMA_CW<0>)) return MOE4_ERR_CUDA;
    return launch<0, EPI_TMA>(ta, tb, td, td, a, st);
}

extern "C" int grouped_expert_gemm_nvfp4_swiglu(const uint8_t *a_codes, const uint8_t *a_sf, const float *a_g_dec,
                                                const uint8_t *b_codes, const uint8_t *b_sf, const float *b_g_dec,
                                                const int32_t *group_offs, int64_t E, int64_t rows_total, int64_t f,
                                                int64_t K, float *gu, uint16_t *h, float *amax_out, uint32_t flags,
                                                void *ws, size_t ws_bytes, void *stream) {
    MOE4_CHECK_ARG(E >= 1 && rows_total >= 0 && rows_total % BM == 0 && f > 0 && f % 128 == 0 && K > 0 &&
                   K % 256 == 0);
    MOE4_CHECK_ARG(a_codes && a_sf && a_g_dec && b_codes && b_sf && b_g_dec && group_offs && gu && h && amax_out);
    MOE4_CHECK_ARG(aligned16(a_codes) && aligned16(b_codes) && aligned16(a_sf) && aligned16(b_sf) && aligned16(gu) &&
                   aligned16(h) && aligned4(amax_out));
    MOE4_CHECK_ARG((flags & ~MOE4_SF_MMA_LAYOUT) == 0);
    const int64_t N = 2 * f;
    MOE4_CHECK_ARG(rows_total < (int64_t(1) << 31) && E * N < (int64_t(1) << 31));
    if (rows_total > 0 && !(flags & MOE4_SF_MMA_LAYOUT) && !scales_ws_ok(rows_total, E * N, K, 16, ws, ws_bytes))
        return MOE4_ERR_WORKSPACE;
    cudaStream_t st = as_stream(stream);
    if (cudaMemsetAsync(amax_out, 0, sizeof(float), st) != cudaSuccess) return MOE4_ERR_CUDA;
    if (rows_total == 0) return MOE4_OK;
    const uint8_t *sfa, *sfb;
    int rc = stage_scales(a_sf, rows_total, b_sf, E * N, K, 16, flags, ws, ws_bytes, &sfa, &sfb, st);
    if (rc != MOE4_OK) return rc;
    CUtensorMap ta, tb;
    // B in 128-row boxes: each tile loads 128 gate rows and the 128 up rows f further on
    if (!make_map(&ta, a_codes, K / 2, rows_total, BM) || !make_map(&tb, b_codes, K / 2, E * N, 128))
        return MOE4_ERR_CUDA;
    Args a{};
    a.sfa = sfa;
    a.sfb = sfb;
    a.a_g_dec = a_g_dec;
    a.b_g_dec = b_g_dec;
    a.offs = group_offs;
    a.E = (int)E;
    a.group_k = 0;
    a.M = rows_total;
    a.N = N;
    a.K = K;
    a.d = gu;
    a.mode = F32;
    a.swiglu_f = f;
    a.h = h;
    a.h_amax = reinterpret_cast<unsigned int *>(amax_out);
    a.n_tiles_n = (int)(f / 128);
    a.n_tiles_m = (int)(rows_total / BM);
    a.num_tiles = (int64_t)a.n_tiles_m * a.n_tiles_n;
    a.sfa_tile_stride = K / 64;
    a.sfb_tile_stride = K / 64;
    CUtensorMap tgu, th;
    if (!make_out_map(&tgu, gu, false, rows_total, N, 32) || !make_out_map(&th, h, true, rows_total, f, 32))
        return MOE4_ERR_CUDA;
    return launch<0, EPI_SWI>(ta, tb, tgu, th, a, st);
}

extern "C" int grouped_expert_gemm_nvfp4_hadamard_mx(const uint8_t *a_codes, const uint8_t *a_sf,
                                                     const float *a_g_dec, const uint8_t *b_codes,
                                                     const uint8_t *b_sf, const float *b_g_dec,
                                                     const int32_t *group_offs, int64_t E, int64_t rows_total,
                                                     int64_t N, int64_t K, uint8_t *q, uint8_t *e8, uint32_t flags,
                                                     void *ws, size_t ws_bytes, void *stream) {
    MOE4_CHECK_ARG(E >= 1 && rows_total >= 0 && rows_total % BM == 0 && N > 0 && N % BN == 0 && K > 0 &&
                   K % 256 == 0);
    MOE4_CHECK_ARG(a_codes && a_sf && a_g_dec && b_codes && b_sf && b_g_dec && group_offs && q && e8);
    MOE4_CHECK_ARG(aligned16(a_codes) && aligned16(b_codes) && aligned16(a_sf) && aligned16(b_sf) && aligned16(q));
    MOE4_CHECK_ARG((flags & ~MOE4_SF_MMA_LAYOUT) == 0);
    MOE4_CHECK_ARG(rows_total < (int64_t(1) << 31) && E * N < (int64_t(1) << 31));
    if (rows_total == 0) return MOE4_OK;
    cudaStream_t st = as_stream(stream);
    const uint8_t *sfa, *sfb;
    int rc = stage_scales(a_sf, rows_total, b_sf, E * N, K, 16, flags, ws, ws_bytes, &sfa, &sfb, st);
    if (rc != MOE4_OK) return rc;
    CUtensorMap ta, tb;
    if (!make_map(&ta, a_codes, K / 2, rows_total, BM) || !make_map(&tb, b_codes, K / 2, E * N, BN))
        return MOE4_ERR_CUDA;
    Args a{};
    a.sfa = sfa;
    a.sfb = sfb;
    a.a_g_dec = a_g_dec;
    a.b_g_dec = b_g_dec;
    a.offs = group_offs;
    a.E = (int)E;
    a.group_k = 0;
    a.M = rows_total;
    a.N = N;
    a.K = K;
    a.d = q;
    a.e8 = e8;
    a.mode = BF16;
    a.n_tiles_n = (int)(N / BN);
    a.n_tiles_m = (int)(rows_total / BM);
    a.num_tiles = (int64_t)a.n_tiles_m * a.n_tiles_n;
    a.sfa_tile_stride = K / 64;
    a.sfb_tile_stride = K / 64;
    return launch<0, EPI_HMX>(ta, tb, ta, tb, a, st);
}

extern "C" int grouped_gemm_mxfp8(const uint8_t *a, const uint8_t *a_e8, const uint8_t *b, const uint8_t *b_e8,
                                  const int32_t *group_offs, int64_t E, int64_t M, int64_t N, int64_t K, void *d,
                                  uint32_t flags, void *ws, size_t ws_bytes, void *stream) {
    MOE4_CHECK_ARG(E >= 1 && M >= 0 && M % BM == 0 && N > 0 && N % BN == 0 && K >= 0 && K % 128 == 0);
    MOE4_CHECK_ARG(a && a_e8 && b && b_e8 && group_offs && d);
    MOE4_CHECK_ARG(aligned16(a) && aligned16(b) && aligned16(a_e8) && aligned16(b_e8) && aligned16(d));
    MOE4_CHECK_ARG((flags & ~(MOE4_OUT_F32 | MOE4_OUT_BF16 | MOE4_SF_MMA_LAYOUT | MOE4_GROUP_M | MOE4_GROUP_K |
                              MOE4_ACCUMULATE)) == 0);
    const bool bf16 = (flags & MOE4_OUT_BF16) != 0;
    MOE4_CHECK_ARG(bf16 != ((flags & MOE4_OUT_F32) != 0));
    const bool gk = (flags & MOE4_GROUP_K) != 0;
    MOE4_CHECK_ARG(gk != ((flags & MOE4_GROUP_M) != 0));
    MOE4_CHECK_ARG(!((flags & MOE4_ACCUMULATE) && bf16));
    MOE4_CHECK_ARG(M < (int64_t(1) << 31) && E * N < (int64_t(1) << 31) && K < (int64_t(1) << 31));
    MOE4_CHECK_ARG(!gk || E * M < (int64_t(1) << 31));  // the output's row coordinate e*M + m is an int32
    cudaStream_t st = as_stream(stream);
    Args g{};
    const uint8_t *sfa, *sfb;
    CUtensorMap ta, tb;
    if (!gk) {
        if (M == 0 || K == 0) return MOE4_OK;
        int rc = stage_scales(a_e8, M, b_e8, E * N, K, 32, flags, ws, ws_bytes, &sfa, &sfb, st);
        if (rc != MOE4_OK) return rc;
        if (!make_map(&ta, a, K, M, BM) || !make_map(&tb, b, K, E * N, BN)) return MOE4_ERR_CUDA;
        g.n_tiles_m = (int)(M / BM);
        g.n_tiles_n = (int)(N / BN);
        g.num_tiles = (int64_t)g.n_tiles_m * g.n_tiles_n;
    } else {
        if (M == 0) return MOE4_OK;
        if (K == 0) {  // every group empty
            if (flags & MOE4_ACCUMULATE) return MOE4_OK;
            return cudaMemsetAsync(d, 0, (size_t)(E * M * N) * (bf16 ? 2 : 4), st) == cudaSuccess ? MOE4_OK
                                                                                              : MOE4_ERR_CUDA;
        }
        int rc = stage_scales(a_e8, M, b_e8, N, K, 32, flags, ws, ws_bytes, &sfa, &sfb, st);
        if (rc != MOE4_OK) return rc;
        if (!make_map(&ta, a, K, M, BM) || !make_map(&tb, b, K, N, BN)) return MOE4_ERR_CUDA;
        g.n_tiles_m = (int)(M / BM);
        g.n_tiles_n = (int)(N / BN);
        g.num_tiles = E * g.n_tiles_m * g.n_tiles_n;
    }
    g.sfa = sfa;
    g.sfb = sfb;
    g.offs = group_offs;
    g.E = (int)E;
    g.group_k = gk;
    g.M = M;
    g.N = N;
    g.K = K;
    g.d = d;
    g.mode = bf16 ? BF16 : ((flags & MOE4_ACCUMULATE) ? ACC_F32 : F32);
    g.sfa_tile_stride = K / 128;
    g.sfb_tile_stride = K / 128;
    if (g.mode == ACC_F32) return launch<1, EPI_REG>(ta, tb, ta, tb, g, st);
    CUtensorMap td;
    if (!make_out_map(&td, d, bf16, gk ? E * M : M, N, TMA_CW<1>)) return MOE4_ERR_CUDA;
    return launch<1, EPI_TMA>(ta, tb, td, td, g, st);
}

extern "C" int grouped_gemm_mxfp8_swiglu_backward(const uint8_t *a, const uint8_t *a_e8, const uint8_t *b,
                                                  const uint8_t *b_e8, const int32_t *group_offs, int64_t E, int64_t M,
                                                  int64_t f, int64_t K, const float *gu, uint16_t *dgu, uint32_t flags,
                                                  void *ws, size_t ws_bytes, void *stream) {
    MOE4_CHECK_ARG(E >= 1 && M >= 0 && M % BM == 0 && f > 0 && f % BN == 0 && K >= 0 && K % 128 == 0);
    MOE4_CHECK_ARG(a && a_e8 && b && b_e8 && group_offs && gu && dgu);
    MOE4_CHECK_ARG(aligned16(a) && aligned16(b) && aligned16(a_e8) && aligned16(b_e8) && aligned16(gu) &&
                   aligned16(dgu));
    MOE4_CHECK_ARG((flags & ~MOE4_SF_MMA_LAYOUT) == 0);
    MOE4_CHECK_ARG(M < (int64_t(1) << 31) && E * f < (int64_t(1) << 31) && K < (int64_t(1) << 31));
    if (M == 0) return MOE4_OK;
    if (M > 0 && K > 0 && !(flags & MOE4_SF_MMA_LAYOUT) && !scales_ws_ok(M, E * f, K, 32, ws, ws_bytes))
        return MOE4_ERR_WORKSPACE;
    cudaStream_t st = as_stream(stream);
    if (K == 0) return MOE4_ERR_UNSUPPORTED;  // an empty contraction: dH = 0, not this kernel's case
    const uint8_t *sfa, *sfb;
    int rc = stage_scales(a_e8, M, b_e8, E * f, K, 32, flags, ws, ws_bytes, &sfa, &sfb, st);
    if (rc != MOE4_OK) return rc;
    CUtensorMap ta, tb, tgu, tdgu;
    if (!make_map(&ta, a, K, M, BM) || !make_map(&tb, b, K, E * f, BN)) return MOE4_ERR_CUDA;
    // GU read and dGU written in 32-row x 16-column chunks
    if (!make_out_map(&tgu, const_cast<float *>(gu), false, M, 2 * f, 16) ||
        !make_out_map(&tdgu, dgu, true, M, 2 * f, 16))
        return MOE4_ERR_CUDA;
    Args g{};
    g.sfa = sfa;
    g.sfb = sfb;
    g.offs = group_offs;
    g.E = (int)E;
    g.group_k = 0;
    g.M = M;
    g.N = f;
    g.K = K;
    g.d = dgu;
    g.mode = BF16;
    g.swb_f = f;
    g.n_tiles_m = (int)(M / BM);
    g.n_tiles_n = (int)(f / BN);
    g.num_tiles = (int64_t)g.n_tiles_m * g.n_tiles_n;
    g.sfa_tile_stride = K / 128;
    g.sfb_tile_stride = K / 128;
    return launch<1, EPI_SWB>(ta, tb, tgu, tdgu, g, st);
}

extern "C" int grouped_gemm_mxfp8_wgrad_sgd(const uint8_t *a, const uint8_t *a_e8, const uint8_t *b,
                                            const uint8_t *b_e8, const int32_t *group_offs, int64_t E, int64_t M,
                                            int64_t N, int64_t K, float *w32, uint16_t *w_bf16, float lr,
                                            float *amax_out, uint32_t flags, void *ws, size_t ws_bytes,
                                            void *stream) {
    MOE4_CHECK_ARG(E >= 1 && M >= 0 && M % BM == 0 && N > 0 && N % BN == 0 && K >= 0 && K % 128 == 0);
    MOE4_CHECK_ARG(a && a_e8 && b && b_e8 && group_offs && w32 && amax_out);
    MOE4_CHECK_ARG(aligned16(a) && aligned16(b) && aligned16(a_e8) && aligned16(b_e8) && aligned16(w32) &&
                   aligned16(w_bf16) && aligned4(amax_out));
    MOE4_CHECK_ARG((flags & ~MOE4_SF_MMA_LAYOUT) == 0);
    MOE4_CHECK_ARG(E * M < (int64_t(1) << 31) && N < (int64_t(1) << 31) && K < (int64_t(1) << 31));
    // a missing workspace is reported before anything is enqueued
    if (M > 0 && K > 0 && !(flags & MOE4_SF_MMA_LAYOUT) && !scales_ws_ok(M, N, K, 32, ws, ws_bytes))
        return MOE4_ERR_WORKSPACE;
    cudaStream_t st = as_stream(stream);
    if (M == 0) {  // empty weight matrices: the amax of every expert that has rows is 0
        sgd_prep_kernel<<<1, 1024, 0, st>>>(group_offs, (int)E, nullptr, reinterpret_cast<unsigned int *>(amax_out));
        return launch_status();
    }
    Args g{};
    const uint8_t *sfa = a_e8, *sfb = b_e8;
    CUtensorMap ta, tb;
    const int64_t Kmap = K > 0 ? K : 128;  // K = 0: every expert is skipped, the maps are never read
    if (K > 0) {
        int rc = stage_scales(a_e8, M, b_e8, N, K, 32, flags, ws, ws_bytes, &sfa, &sfb, st);
        if (rc != MOE4_OK) return rc;
    }
    constexpr int BNS = EpiCfg<EPI_SGD>::BNT;
    static_assert(EpiCfg<EPI_SGD32>::BNT == BNS, "both SGD modes use the same tiles");
    if (!make_map(&ta, a, Kmap, M, BM) || !make_map(&tb, b, Kmap, N, BNS)) return MOE4_ERR_CUDA;
    // the expert order for the tile schedule, after the staged scales in the workspace (without
    // room for it the tiles run in expert order); the same one-CTA kernel clears the amax of the
    // experts that have rows
    size_t used = 0;
    if (K > 0 && !(flags & MOE4_SF_MMA_LAYOUT)) {
        const size_t na = (size_t)(M * (K / 32)), nb = (size_t)(N * (K / 32));
        used = (na + 255) / 256 * 256 + (nb + 255) / 256 * 256;
    }
    int32_t *order = nullptr;
    if (E < 4096 && ws && aligned16(ws) && ws_bytes >= used + (size_t)(E + 1) * sizeof(int32_t))
        order = reinterpret_cast<int32_t *>(static_cast<uint8_t *>(ws) + used);
    sgd_prep_kernel<<<1, 1024, 0, st>>>(group_offs, (int)E, order, reinterpret_cast<unsigned int *>(amax_out));
    g.order = order;
    g.sfa = sfa;
    g.sfb = sfb;
    g.offs = group_offs;
    g.E = (int)E;
    g.group_k = 1;
    g.M = M;
    g.N = N;
    g.K = K;
    g.d = w32;
    g.mode = SGD;
    g.w_bf16 = w_bf16;
    g.lr = lr;
    g.amax = reinterpret_cast<unsigned int *>(amax_out);
    g.n_tiles_m = (int)(M / BM);
    g.n_tiles_n = (int)(N / BNS);
    g.num_tiles = E * g.n_tiles_m * g.n_tiles_n;
    g.sfa_tile_stride = K / 128;
    g.sfb_tile_stride = K / 128;
    CUtensorMap tw, twb;  // the master weights and their bf16 copy as [E*M, N], 16-column x 32-row boxes
    if (!make_map_t(&tw, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 4, w32, N, E * M, SGD_CW, 32, CU_TENSOR_MAP_SWIZZLE_64B))
        return MOE4_ERR_CUDA;
    if (!w_bf16)
        twb = tw;  // never used: the bf16 copy is not written
    else if (!make_map_t(&twb, CU_TENSOR_MAP_DATA_TYPE_UINT16, 2, w_bf16, N, E * M, SGD_CW, 32,
                         CU_TENSOR_MAP_SWIZZLE_32B))
        return MOE4_ERR_CUDA;
    return w_bf16 ? launch<1, EPI_SGD>(ta, tb, tw, twb, g, st) : launch<1, EPI_SGD32>(ta, tb, tw, twb, g, st);
}

template <int KIND, bool kCopySf>
static int launch_peak(int64_t iters, int64_t ctas, uint32_t *sink, cudaStream_t st) {
    constexpr int SMEM = A_TILE + BN * BKB + 3 * 4 * 512 + 64 + 1024;
    if (cudaFuncSetAttribute(mma_peak_kernel<KIND, kCopySf>, cudaFuncAttributeMaxDynamicSharedMemorySize, SMEM) !=
        cudaSuccess)
        return MOE4_ERR_CUDA;
    mma_peak_kernel<KIND, kCopySf><<<(unsigned)ctas, 128, SMEM, st>>>(iters, sink);
    return launch_status();
}

extern "C" int moe4_tensor_peak_probe(int kind, int64_t iters, int64_t ctas, uint32_t *sink, void *stream) {
    MOE4_CHECK_ARG(kind >= 0 && kind <= 3 && iters >= 1 && iters <= (int64_t(1) << 20) && ctas >= 1 && ctas <= 4096);
    MOE4_CHECK_ARG(sink && aligned4(sink));
    cudaStream_t st = as_stream(stream);
    switch (kind) {
        case 0: return launch_peak<0, false>(iters, ctas, sink, st);
        case 1: return launch_peak<1, false>(iters, ctas, sink, st);
        case 2: return launch_peak<0, true>(iters, ctas, sink, st);
        default: return launch_peak<1, true>(iters, ctas, sink, st);
    }
}

extern "C" int moe4_selftest_wait(int64_t limit_cycles, void *stream) {
    MOE4_CHECK_ARG(limit_cycles > 0 && limit_cycles <= (int64_t(1) << 32));
    wait_selftest_kernel<<<1, 32, 0, as_stream(stream)>>>((long long)limit_cycles);
    return launch_status();
}
