// tl_gemm.h -- internal interface of the three tile GEMMs (host side).
//
//   forward  (K1): Y_i  = X . W_i          A = X  (K-major), B = W_i (N-major)
//   weight   (K3): dW_i = X^T . dY_i       A = X^T (M-major), B = dY_i (N-major)
//   input    (K2): dX  (+)= dY_i . W_i^T   A = dY_i (K-major), B = W_i^T (K-major)
//
// All three run one persistent kernel template: bf16 operands fed by TMA into
// a shared-memory ring, tcgen05 MMAs accumulating in fp32 in tensor memory,
// and an epilogue that rounds to bf16 (K1, K3) or stores / adds fp32 (K2).
// K2 may also round to bf16, after adding an fp32 addend: the last dX launch
// of an operator in a chain writes the previous operator's dY directly.
#pragma once
#include <cstdint>
#include <string>
#include <cuda_runtime.h>

namespace tl {

enum class OutKind : int { BF16 = 0, F32 = 1 };

// D[m_dim, n_dim] (ld ldd) = sum_k A[m, k] B[k, n] over k < k_dim.
// A is given either K-major (a_ptr[m * lda + k]) or M-major (a_ptr[k * lda + m]);
// B either K-major (b_ptr[n * ldb + k]) or N-major (b_ptr[k * ldb + n]).
struct GemmDesc {
    int64_t m_dim = 0, n_dim = 0, k_dim = 0;
    const void* a = nullptr;
    int64_t lda = 0;
    bool a_mn_major = false;
    const void* b = nullptr;
    int64_t ldb = 0;
    bool b_mn_major = false;
    // Optional further B segments (K-major B only): with nseg > 1, reduction
    // rows [j k_seg, (j+1) k_seg) are read from segment j, bseg[j][n * ldb +
    // (k - j k_seg)], where bseg[0] is b.  k_seg is a multiple of kBlockK and
    // nseg * k_seg == k_dim.  Lets one launch reduce over several weight
    // tiles that sit in different ring slots.
    static constexpr int kMaxSeg = 4;
    const void* bseg[kMaxSeg] = {};
    int32_t nseg = 1;
    int64_t k_seg = 0;
    void* d = nullptr;
    int64_t ldd = 0;
    OutKind out = OutKind::BF16;
    bool accumulate = false;  // F32 only: D += A.B
    // BF16 output of the input-gradient kind (A and B K-major) only: with an
    // addend, D = bf16(addend + A.B), addend fp32 [m_dim][ld_addend], the sum
    // taken in fp32 and rounded once.
    const float* addend = nullptr;
    int64_t ld_addend = 0;
    int32_t* err = nullptr;   // device word for bounded-wait timeouts
    // Device word the CTAs draw output tiles from (dynamic schedule); zero
    // before the launch, and left zero by a launch that completes without a
    // timeout.  nullptr: a static round-robin schedule.
    uint32_t* tile_counter = nullptr;
    uint64_t timeout_ns = 2000000000ull;  // limit of every bounded wait
    bool withhold_loads = false;  // failure-path self-test: the producer issues no loads
};

// Shape / alignment rules shared by the launcher and the ABI checks.
// Returns an empty string if `g` can be launched, else the reason.
std::string gemm_check(const GemmDesc& g);

// Enqueue one GEMM on `stream`.  num_sms bounds the persistent grid.
cudaError_t gemm_launch(const GemmDesc& g, int num_sms, cudaStream_t stream, std::string* why);

// Shared host helpers (defined in tl_gemm.cu).
void choose_tile_order(int64_t k_dim, int tile_m, int num_m, int num_n, int concurrent, int32_t* raster,
                       int32_t* group, int32_t* stream_shared);
bool cta_pair_enabled();

// Tile shape of the kernel (exported for sizing and tests).
constexpr int kBlockM = 128;
constexpr int kBlockN = 256;
constexpr int kBlockK = 64;

// Error bits a kernel ORs into *err when a bounded wait gives up.
enum : int32_t {
    kErrProducerWait = 1,
    kErrMmaWaitFull = 2,
    kErrMmaWaitTmem = 4,
    kErrEpilogueWait = 8,
    kErrDrainWait = 16,
    kErrTileQueueWait = 64,  // a role gave up waiting for the next tile of the dynamic schedule
};

}  // namespace tl
