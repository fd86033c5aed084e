// SpGEMM internals shared by spgemm.cu (kernels) and api.cu (handle).
#pragma once

#include "internal.cuh"

namespace lbcsr {

// ---------------------------------------------------------------- SpGEMM
// C = A * B (A m-by-k, B k-by-n, CSR), OpSparse's two phases.  Rows of C
// are binned by their products (the sum over the row of A of the lengths
// of the rows of B it picks): bins of at most 16, 128, 512, 1024, 2048 and
// 4096 products, then the rest (the dense bin); bin_rows holds the
// rows of bin 0, then bin 1, ... each in increasing order.  The last bin is
// the dense one.
constexpr int kSpgemmBins = 7;
struct SpgemmArgs {
    int32_t m, n;
    const int32_t *a_ptr, *a_col, *b_ptr, *b_col;
    int64_t *products;     // [m]
    int32_t *bin_rows;     // [m]
    int64_t bin_count[kSpgemmBins];  // host copy, read back after the analysis
    const int32_t *num_bin_rows;     // [m] the numeric phase's bins (by entries of C)
    int64_t num_bin_count[kSpgemmBins];
    int64_t *row_nnz;      // [m + 1]  entries of each row of C (symbolic phase)
    int64_t *c_ptr;        // [m + 1]  their exclusive prefix sum
    // the dense bin: entry space, pieces, waves and the slots of a wave
    int64_t dense_slots;     // rows of C held at once (a wave)
    const int64_t *dense_e_off, *dense_pp, *dense_piece_k0, *dense_piece_e;
    const int32_t *dense_piece_row;
    int64_t dense_waves;
    const int64_t *h_wave_row;    // HOST [waves + 1]: first dense row of each wave
    const int64_t *h_wave_piece;  // HOST [waves + 1]: first piece of each wave
    unsigned *dense_bits;     // [dense_slots * spgemm_bit_words(n)], zero between uses
    void *dense_vals;         // [dense_slots * n] value type, zero between uses
    int64_t dense_segs;       // column segments per dense row (spgemm_segments)
    int64_t *dense_seg_cnt;   // [dense rows * segs] zero before the symbolic phase
    int64_t *dense_seg_off;   // [dense rows * segs + 1]
    int64_t *dense_seg_scan;  // scan scratch for them
    int32_t *error;        // bit 1: a row of C outgrew its symbolic size
};
int64_t spgemm_chunks(int32_t m);  // classification chunks; counts/offsets hold kSpgemmBins * chunks (+1)
int64_t spgemm_piece_products();  // products per piece of the dense bin
int64_t spgemm_segments(int32_t n);  // column segments per dense row when it is read back
int64_t spgemm_bit_words(int32_t n);  // words of bits per dense row (padded for 16-byte loads)
// dense bin layout: alen[j] (scratch) and e_off[0..nrows] = entries of A before dense row j
cudaError_t launch_spgemm_dense_layout(const SpgemmArgs &a, const int32_t *drows, int64_t nrows, int64_t *alen,
                                       int64_t *e_off, int64_t *scan_scratch, cudaStream_t stream);
// blen[e] (scratch), pp[0..entries] = products before entry e, rowp[0..nrows] = pp[e_off[j]]
cudaError_t launch_spgemm_dense_products(const SpgemmArgs &a, const int32_t *drows, int64_t nrows,
                                         const int64_t *e_off, int64_t entries, int64_t *blen, int64_t *pp,
                                         int64_t *rowp, int64_t *scan_scratch, cudaStream_t stream);
// piece_e[c] = last entry e with pp[e] <= piece_k0[c]
cudaError_t launch_spgemm_dense_locate(int64_t pieces, const int64_t *piece_k0, const int64_t *pp, int64_t entries,
                                       int64_t *piece_e, cudaStream_t stream);
// products, bin_count (device, chunk_counts / chunk_offsets), bin_rows
cudaError_t launch_spgemm_analysis(const SpgemmArgs &a, int64_t *chunk_counts, int64_t *chunk_offsets,
                                   int64_t *scan_scratch, cudaStream_t stream);
// bins for the numeric phase, after the symbolic one: key (scratch, [m]) =
// the products for rows of at most 16 or more than 4096 products, else the
// row's entries; rows written to num_bin_rows; counts per [bin][chunk] as
// for launch_spgemm_analysis
cudaError_t launch_spgemm_numeric_bins(const SpgemmArgs &a, int64_t *key, int64_t *chunk_counts,
                                       int64_t *chunk_offsets, int64_t *scan_scratch, int32_t *num_bin_rows,
                                       cudaStream_t stream);
// row_nnz and c_ptr (needs bin_count and the dense scratch)
cudaError_t launch_spgemm_symbolic(spmv_dtype_t dtype, const SpgemmArgs &a, int64_t *scan_scratch,
                                   cudaStream_t stream);
// c_col, c_val (each row by increasing column) and c_row_ptr (int32) when non-null
cudaError_t launch_spgemm_numeric(spmv_dtype_t dtype, const SpgemmArgs &a, const void *a_val, const void *b_val,
                                  int32_t *c_row_ptr, int32_t *c_col, void *c_val, cudaStream_t stream);

}  // namespace lbcsr
