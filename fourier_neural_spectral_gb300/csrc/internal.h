// internal.h -- plan object and kernel launchers shared by the host files of
// libfnospec.  Not part of the public ABI (that is include/fnospec.h).
#pragma once

#include <vector>

#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

#include "common.cuh"
#include "fnospec.h"

// Bits of the device error word.
enum : unsigned {
    FNO_DEVERR_BOUNDS = 1u << 0,   // an index check in a kernel failed
    FNO_DEVERR_TIMEOUT = 1u << 1,  // a bounded wait gave up
};

struct fno_kernel_desc {
    char name[48];
    size_t bytes;   // algorithmic bytes (compulsory reads + writes)
    size_t flops;   // algorithmic flops
};

// Optional per-kernel event recording during one execute.
struct fno_launch_ctx {
    cudaEvent_t* events = nullptr;
    int count = 0;
    int next = 0;
    cudaError_t mark(cudaStream_t s) {
        if (!events || next >= count) return cudaSuccess;
        return cudaEventRecord(events[next++], s);
    }
};

// Dynamic shared memory one block may ask for: the opt-in limit (227 KB), less
// room for the static shared memory (the output ranges) that range-checked
// builds add to their kernels.
#ifdef FNO_DEBUG
constexpr size_t kMaxDynSmem = 227 * 1024 - 1024;
#else
constexpr size_t kMaxDynSmem = 227 * 1024;
#endif

// The output ranges a range-checked build checks a launch's stores against:
// FNO_DBG_ARG1(ptr, bytes, plan) for one output, FNO_DBG_ARG2 for two.  The
// first range is shortened by the plan's debug margin (the test hook that
// makes the last outputs count as out of range).  Empty without FNO_DEBUG.
#ifdef FNO_DEBUG
#define FNO_DBG_RANGES2(p0, n0, p1, n1, plan)                                                \
    fno::fno_dbg_ranges {                                                                     \
        {((const char*)(const void*)(p0)), ((const char*)(const void*)(p1))},             \
            {((const char*)(const void*)(p0)) +                                              \
                 ((size_t)(n0) > (plan).dbg_margin ? (size_t)(n0) - (plan).dbg_margin : 0),  \
             ((const char*)(const void*)(p1)) + (n1)},                                      \
            (plan).err                                                                        \
    }
#define FNO_DBG_ARG2(p0, n0, p1, n1, plan) , FNO_DBG_RANGES2(p0, n0, p1, n1, plan)
#define FNO_DBG_ARG1(p0, n0, plan) FNO_DBG_ARG2(p0, n0, nullptr, 0, plan)
#else
#define FNO_DBG_ARG2(p0, n0, p1, n1, plan)
#define FNO_DBG_ARG1(p0, n0, plan)
#endif

// Launch with programmatic stream serialisation (the kernel must call
// griddep_wait() before touching memory that earlier kernels of the stream
// write, then griddep_launch_dependents(); see common.cuh).
template <typename... KArgs, typename... Args>
cudaError_t launch_pdl(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem,
                       cudaStream_t s, Args&&... args) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kernel, static_cast<KArgs>(args)...);
}

constexpr int kMaxKernels = 8;

struct fno_plan_s {
    int B, Cin, Cout, H, W, m1, m2;
    int dims;               // 2, or 1 for the 1D layer (H = 1, W = L, m1 = 0, m2 = m)
    int nm;                 // retained modes per plane: 2*m1*m2 (m2 for the 1D layer)
    fno_precision_t prec;
    int device;
    int sms;                // multiprocessors of the device (persistent grids)
    float scale;            // 1/sqrt(H*W), rounded once from double
    float2* tw_h;           // e^{+2 pi i j / H}, j in [0, H)
    float2* tw_w;           // e^{+2 pi i j / W}, j in [0, W)
    float* g_irows;         // direct-DFT inverse rows: twiddle tiles (dft_irows_table), or null
    float* g_frows;         // direct-DFT forward rows: twiddle tiles (dft_frows_table), or null
    float2* g_cols;         // direct-DFT column steps: twiddle matrices (dft_cols_table), or null
    unsigned* err;          // device error word
    unsigned long long* gbar;  // grid-barrier counter of the single-launch layer
    int single_launch;      // execute runs the whole layer as one launch
    size_t dbg_margin;      // range-checked builds: bytes taken off each launch's first
                            // output range (fno_plan_debug_bounds_margin)
    // workspace layout (byte offsets, each 256-byte aligned)
    size_t off_X, off_Z, off_T, ws_bytes;
    int path;               // 0: shape-generic kernels, 1: fused transform kernels
    int mix_path;           // 0: mix_fma, 1: mix_tma, 2: mix_tc (tcgen05), 3: mix_wide,
                            // 4: mix_adj_fma (adjoint plans only), 5: mix_tcm (tcgen05,
                            // weights in tensor memory)
    bool adjoint;           // contraction with w conjugated and transposed (backward's
                            // plan: Cin, Cout are w's Cout, Cin)
    fno_plan_s* adj;        // the backward's plan (channels swapped), owned
    bool shares_tables;     // tw_h, tw_w and err belong to the parent plan
    int tc_split;           // mix_tc, mix_tcm: 1 (TF32) or 3 (split TF32, hi*hi + hi*lo + lo*hi)
    int R, P;               // fused path, forward: column length per CTA and H / R
    int Ri, Pi;             // fused path, inverse: the same
    int launches;           // kernel launches per execute
    fno_kernel_desc kernels[kMaxKernels];
    cudaEvent_t* events;    // armed per-kernel timing events (count = launches + 1)
    int nevents;
    char desc[256];
};

// One-time kernel attribute set-up (dynamic shared memory limits).
cudaError_t stages_generic_init();
cudaError_t mix_init();

// Fused transform kernels (stages_fused.cu).
cudaError_t stages_fused_init();
bool fused_supported(int W, int H, int m1, int m2, int* R_fwd, int* R_inv);
size_t fused_smem_bytes_any(int W, int R, int m2);
cudaError_t launch_forward_fused(const fno_plan_s& p, const float* x, float2* X, cudaStream_t s,
                                 fno_launch_ctx* ctx);
cudaError_t launch_inverse_fused(const fno_plan_s& p, const float2* Z, float* y, cudaStream_t s,
                                 fno_launch_ctx* ctx);
// Long-row variants (stages_big.cu), W in {512, 1024, 2048, 4096}, m2 <= 64.
cudaError_t stages_big_init();
size_t big_smem_bytes_any(int W, int R, int m2, bool fwd);
bool big_z_staged_any(int W, int R, int m1, int m2);
cudaError_t launch_forward_big(const fno_plan_s& p, const float* x, float2* X, cudaStream_t s);
cudaError_t launch_inverse_big(const fno_plan_s& p, const float2* Z, float* y, cudaStream_t s);
// the 1D layer's row transforms on the long-row kernels (W = 512 .. 4096, m2 <= 64)
bool rows1d_supported(int W, int m2);
cudaError_t launch_forward_rows1d(const fno_plan_s& p, const float* x, float2* X, cudaStream_t s,
                                  fno_launch_ctx* ctx);
cudaError_t launch_inverse_rows1d(const fno_plan_s& p, const float2* Z, float* y, cudaStream_t s,
                                  fno_launch_ctx* ctx);

// TMA-fed fp32 contraction (mix_tma.cu).
cudaError_t mix_tma_init();
bool mix_tma_supported(int B, int Cin, int Cout, int nm);
cudaError_t launch_mix_tma(const fno_plan_s& p, const float2* X, const float2* w, float2* Z,
                           cudaStream_t s, fno_launch_ctx* ctx);

// fp32 contraction over blocks of 32 consecutive modes (mix_wide.cu).
cudaError_t mix_wide_init();
bool mix_wide_supported(int B, int Cin, int Cout, int nm);
bool wgrad_wide_supported(int nm);
// after_own_forward: the kernel just before this one is the library's forward
// stage (w may then be fetched before the programmatic-launch wait).
cudaError_t launch_mix_wide(const fno_plan_s& p, const float2* X, const float2* w, float2* Z,
                            bool after_own_forward, cudaStream_t s, fno_launch_ctx* ctx);
cudaError_t launch_wgrad_wide(const fno_plan_s& p, const float2* X, const float2* G, float2* gw,
                              cudaStream_t s);

// FNO block epilogue (block.cu).
cudaError_t block_init();
bool block_supported(int Cin);
cudaError_t block_tc_init();
bool block_tc_supported(int Cin, int Cout);
cudaError_t launch_block_tc(const fno_plan_s& p, const float* x, const float* w_pw,
                            const float* bias, int act, float* y, bool after_own_inverse,
                            cudaStream_t s);
cudaError_t launch_block_epilogue(const fno_plan_s& p, const float* x, const float* w_pw,
                                  const float* bias, int act, float* y, bool after_own_inverse,
                                  cudaStream_t s);

// Backward-only kernels (backward.cu).
cudaError_t launch_wgrad(const float2* X, const float2* G, float2* gw, int B, int Cin, int Cout,
                         int nm, int m2, int W, cudaStream_t s);
cudaError_t launch_mix_adjoint_fma(const fno_plan_s& p, const float2* G, const float2* w,
                                   float2* GX, cudaStream_t s, fno_launch_ctx* ctx);

// tcgen05 tensor-core contraction (mix_tc.cu).
cudaError_t mix_tc_init();
bool mix_tc_supported(int B, int Cin, int Cout, int nm, int split);
cudaError_t launch_mix_tc(const fno_plan_s& p, const float2* X, const float2* w, float2* Z,
                          int split, cudaStream_t s, fno_launch_ctx* ctx);

// tcgen05 contraction with the weight operand in tensor memory (mix_tcm.cu):
// 8 modes x 64 output channels per CTA, batch up to 16.
cudaError_t mix_tcm_init();
bool mix_tcm_supported(int B, int Cin, int Cout, int nm);
cudaError_t launch_mix_tcm(const fno_plan_s& p, const float2* X, const float2* w, float2* Z,
                           int split, bool after_own_forward, cudaStream_t s,
                           fno_launch_ctx* ctx);

// The whole layer in one cooperative launch (layer_persistent.cu).
cudaError_t layer_persistent_init();
bool layer_persistent_supported(const fno_plan_s& p);
cudaError_t launch_layer_persistent(const fno_plan_s& p, const float* x, const float2* w,
                                    float* y, float2* X, float2* Z, cudaStream_t s,
                                    fno_launch_ctx* ctx);

// Direct-DFT transforms for H or W not a power of two (stages_dft.cu); the
// shape-generic launchers below route such shapes there.
bool dft_path(int H, int W);
// Twiddle tiles of the direct-DFT inverse row step for rows of W points and m2
// retained columns (empty when that step does not use them), in the layout
// dft_irows_kernel streams: [pass][4 shifts][2*m2][64] floats.
std::vector<float> dft_irows_table(int W, int m2, double scale);
// The same for the forward row step ([pass][4 shifts][64][NP] floats, NP = 2*m2
// rounded up to 8, 16, 24 or 32; empty above 32).
std::vector<float> dft_frows_table(int W, int m2, double scale);
// The column steps' twiddle matrices for columns of H points and 2*m1 retained
// rows k1(r): the forward's At[h][r] = e^{-2 pi i k1(r) h / H} (H x 2m1) followed
// by the inverse's At[r][h] = e^{+2 pi i k1(r) h / H} (2m1 x H).
std::vector<float2> dft_cols_table(int H, int m1);
cudaError_t stages_dft_init();
cudaError_t launch_forward_dft(const fno_plan_s& p, const float* x, float2* X, float2* T,
                               cudaStream_t s, fno_launch_ctx* ctx);
cudaError_t launch_inverse_dft(const fno_plan_s& p, const float2* Z, float* y, float2* T,
                               cudaStream_t s, fno_launch_ctx* ctx);
cudaError_t launch_forward_1d(const fno_plan_s& p, const float* x, float2* X, cudaStream_t s,
                              fno_launch_ctx* ctx);
cudaError_t launch_inverse_1d(const fno_plan_s& p, const float2* Z, float* y, cudaStream_t s,
                              fno_launch_ctx* ctx);

// Stage launchers (all asynchronous on stream s).
// Each launcher calls ctx->mark(s) after every kernel it enqueues.
cudaError_t launch_forward_modes(const fno_plan_s& p, const float* x, float2* X, float2* T,
                                 cudaStream_t s, fno_launch_ctx* ctx);
cudaError_t launch_mix_modes(const fno_plan_s& p, const float2* X, const float2* w, float2* Z,
                             cudaStream_t s, fno_launch_ctx* ctx);
cudaError_t launch_inverse_modes(const fno_plan_s& p, const float2* Z, float* y, float2* T,
                                 cudaStream_t s, fno_launch_ctx* ctx);
