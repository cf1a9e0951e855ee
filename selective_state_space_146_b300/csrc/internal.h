// internal.h -- host-side declarations shared by the library's translation
// units (not part of the public ABI).
#pragma once
#include <cstdint>
#include <cuda.h>
#include <cuda_runtime.h>

#include "ssscan.h"

namespace ss {

// Host view of one selective-scan call, element strides.
struct ScanArgs {
    int Bsz, D, N, L;
    int dtype;  // SS_F32 / SS_BF16
    const void* u;  int64_t su_b, su_d, su_t;
    const void* dl; int64_t sdl_b, sdl_d, sdl_t;
    const void* z;  int64_t sz_b, sz_d, sz_t;
    void* y;        int64_t sy_b, sy_d, sy_t;
    const void* Bm; int64_t sB_b, sB_n, sB_t;
    const void* Cm; int64_t sC_b, sC_n, sC_t;
    // B, C per channel group: G groups of D / G consecutive channels, group
    // stride sB_g / sC_g; G <= 1 is one B, C per batch row
    int G; int64_t sB_g, sC_g;
    const float* A; int64_t sA_d, sA_n;
    const float* Dv; int64_t sD;
    const float* bias; int64_t sbias;
    float* last; int64_t sl_b, sl_d, sl_n;
    const float* h0; int64_t sh_b, sh_d, sh_n;  // initial state, may be null
    // causal conv1d + SiLU in front of the scan (u holds its input x); cw null = off
    const float* cw; int64_t scw_d, scw_k;
    const float* cb; int64_t scb;
    int cwidth;
    int softplus;
    unsigned* err;  // device error word
    // state at the start of every 8-step sub-chunk, [b][d][ceil(L/8)][16]
    // fp32, written by the forward when non-null (the backward's layout)
    float* ckpt = nullptr;
};

// Host view of one SSD call, element strides.
struct SSDArgs {
    int Bsz, L, H, P, G, N, chunk;
    int dtype;
    const void* x;  int64_t sx_b, sx_l, sx_h, sx_p;
    const void* dt; int64_t sdt_b, sdt_l, sdt_h;
    const float* A; int64_t sA;
    const void* Bm; int64_t sB_b, sB_l, sB_g, sB_n;
    const void* Cm; int64_t sC_b, sC_l, sC_g, sC_n;
    const float* Dv; int64_t sD;
    void* y;        int64_t sy_b, sy_l, sy_h, sy_p;
    float* last;    int64_t sl_b, sl_h, sl_p, sl_n;
    const float* h0; int64_t sh_b, sh_h, sh_p, sh_n;  // initial state, may be null
    unsigned* err;
};

// One recurrent step of the selective scan (decode), element strides.
struct StepArgs {
    int Bsz, D, N, dtype;
    float* state; int64_t ss_b, ss_d, ss_n;
    const void* u; int64_t su_b, su_d;
    const void* dl; int64_t sdl_b, sdl_d;
    const void* z; int64_t sz_b, sz_d;
    void* y; int64_t sy_b, sy_d;
    const void* Bm; int64_t sB_b, sB_n;
    const void* Cm; int64_t sC_b, sC_n;
    const float* A; int64_t sA_d, sA_n;
    const float* Dv; int64_t sD;
    const float* bias; int64_t sbias;
    int softplus;
};

// One recurrent step of the SSD scan (decode), element strides.
struct SSDStepArgs {
    int Bsz, H, P, G, N, dtype;
    float* state; int64_t ss_b, ss_h, ss_p, ss_n;
    const void* x; int64_t sx_b, sx_h, sx_p;
    const void* dt; int64_t sdt_b, sdt_h;
    const float* A; int64_t sA;
    const void* Bm; int64_t sB_b, sB_g, sB_n;
    const void* Cm; int64_t sC_b, sC_g, sC_n;
    const float* Dv; int64_t sD;
    void* y; int64_t sy_b, sy_h, sy_p;
};

// Backward of the selective scan, element strides.  The fp32 gradients dA
// (D, N), dB and dC (Bsz, N, L), dD and dbias (D) are contiguous.
struct BwdArgs {
    int Bsz, D, N, L, dtype;
    const void* u;    int64_t su_b, su_d, su_t;
    const void* dl;   int64_t sdl_b, sdl_d, sdl_t;
    const void* z;    int64_t sz_b, sz_d, sz_t;
    const void* dout; int64_t sg_b, sg_d, sg_t;
    const void* Bm;   int64_t sB_b, sB_n, sB_t;
    const void* Cm;   int64_t sC_b, sC_n, sC_t;
    const float* A;   int64_t sA_d, sA_n;
    const float* Dv;  int64_t sD;
    const float* bias; int64_t sbias;
    int softplus;
    void* du;  int64_t sdu_b, sdu_d, sdu_t;
    void* ddl; int64_t sddl_b, sddl_d, sddl_t;
    void* dz;  int64_t sdz_b, sdz_d, sdz_t;
    float *dA, *dB, *dC, *dD, *dbias;
    float* ckpt;  // chunk-start states, filled by the kernel
    unsigned* err;
    // the forward's states at every 8-step sub-chunk start, [b][d][ceil(L/8)][16]
    // (ss_selective_scan_fwd_ckpt); when given the backward skips its forward pass
    const float* ckpt_in = nullptr;
};

// Scratch provider: either stream-ordered allocation or a fixed buffer.
struct Scratch {
    void* (*alloc)(size_t bytes, cudaStream_t st, void* ctx);
    void (*release)(void* p, cudaStream_t st, void* ctx);
    void* ctx;
    size_t limit = ~size_t(0);  // largest request alloc can meet (kernels size to fit)
};

// Row copies between a caller's strided rows of L elements and a padded
// layout (row pitch Lp elements, Lp * element size a multiple of 16 bytes) in
// scratch, for calls whose rows the TMA kernels cannot map.  Copies are
// gathered and go out together, up to kMaxRowCopies per launch (one block
// row copy at a time, coalesced whatever the rows' alignment).
constexpr int kMaxRowCopies = 8;
struct RowCopyList {
    const void* src[kMaxRowCopies];
    void* dst[kMaxRowCopies];
    int64_t ss0[kMaxRowCopies], ss1[kMaxRowCopies], ds0[kMaxRowCopies], ds1[kMaxRowCopies];
    int64_t rows[kMaxRowCopies];
    int n1[kMaxRowCopies];
    int count, L;
};
class RowPacker {
  public:
    RowPacker(int dtype, int64_t L, int64_t Lp, cudaStream_t st);
    // rows (i, j), i < n0 at element stride s0 and j < n1 at stride s1, of
    // `other`, into `padded` (row i * n1 + j at pitch Lp) when `in`, else from
    // `padded` back into `other`; a null `other` is skipped
    void add(void* padded, const void* other, int64_t n0, int64_t s0, int64_t n1, int64_t s1,
             bool in);
    // launches what was added; SS_OK or SS_ERR_LAUNCH (which sticks)
    int flush();
    int status() const { return rc_; }

  private:
    RowCopyList list_{};
    int dtype_;
    int64_t Lp_, max_rows_ = 0;
    cudaStream_t st_;
    int rc_ = 0;
};
// Padded length for rows of L elements: the row pitch rounded up to 16 bytes.
inline int64_t padded_len(int64_t L, int es) { return (L * es + 15) / 16 * 16 / es; }

int launch_selective(const ScanArgs& a, cudaStream_t st, const Scratch& scratch);
// scan_seq (N = 16, fast layouts, with or without the conv in front, no
// checkpoints); *taken is false when the call does not fit it.
int launch_selective_seq(const ScanArgs& a, cudaStream_t st, const Scratch& scratch, bool* taken);
// Unit t-stride, 16-byte aligned rows and strides, N = 16: the TMA kernels' layout.
bool fast_layout_ok(const ScanArgs& a);
// A diagnostic switch set by ss_debug_set_path (SS_DEBUG_*), -1 when unset.
int debug_path(int which);
int launch_ssd(const SSDArgs& a, cudaStream_t st, const Scratch& scratch);
// B, C per small channel group (scan_pc / scan_pc_tma); *taken is false when
// the layout suits neither and the caller should run the general kernel.
int launch_selective_grouped(const ScanArgs& a, cudaStream_t st, bool* taken);
// N in {32, 64, 128} with B, C shared per batch row (scan_wide); *taken is
// false when the shape or layout does not fit and the general kernel runs.
int launch_selective_wide(const ScanArgs& a, cudaStream_t st, bool* taken);
// A kernel whose bounded wait always runs out (ss_selftest_timeout).
int launch_selftest_wait(unsigned limit_us, unsigned* err, cudaStream_t st);
// ex2.approx.f32 operations per SM per clock (ss_probe_ex2_rate); synchronises st.
int probe_ex2_rate(double* per_sm_clk, cudaStream_t st);
// channel-steps per second of the sequential and the warp-shuffle scan forms
// (ss_probe_scan_forms); synchronises st.
int probe_scan_forms(double* seq_steps_per_s, double* shfl_steps_per_s, cudaStream_t st);
int launch_selective_bwd(const BwdArgs& a, cudaStream_t st, const Scratch& scratch);
int launch_selective_step(const StepArgs& a, cudaStream_t st);
int launch_ssd_step(const SSDStepArgs& a, cudaStream_t st);

// Counts kernels launched by the library.
void count_launch(int n);
int sm_count_current();
// cuTensorMapEncodeTiled resolved through the runtime (no libcuda link).
void* tensor_map_encoder();
// Tensor map of a (Bsz, D, L) activation (or (Bsz, N, L) B / C) with unit
// t-stride: box of box_t steps x box_d rows, 128-byte swizzle if `swizzle`.
bool make_map_3d(CUtensorMap* m, const void* base, int dtype, int64_t L, int64_t D, int64_t Bsz,
                 int64_t sd, int64_t sb, int box_t, int box_d, bool swizzle = true);
// The same with the swizzle span given in bytes (0, 64 or 128).
bool make_map_3d_sw(CUtensorMap* m, const void* base, int dtype, int64_t L, int64_t D, int64_t Bsz,
                    int64_t sd, int64_t sb, int box_t, int box_d, int swizzle_bytes);

}  // namespace ss
