/*
 * tq_oracle.h -- plain fp64 CPU oracle of the quantised (TurboQuant) KV cache.
 *
 * TEST INFRASTRUCTURE ONLY, like hfa_oracle.h: loaded by the test suite and the
 * benchmark's CPU leg, never by the CUDA library, sharing no code, table or helper
 * with it.
 *
 * Source: hf2q documentation page "gemma4/gpu_full_attn.rs", encode_one_layer: the
 * Hadamard-quantize KV encode (hadamard_quantize_kv, _hb: sign pre-multiply, normalised
 * FWHT, a per-block norm -- one per 256 dims, two for a 512-wide head -- and Lloyd-Max
 * codes, 4-bit nibble-packed, or one byte per element at 5, 6 and 8 bits), the TQ attention
 * (flash_attn_vec_tq / _tq_hb: Q pre-rotated by the same sign pre-multiply and FWHT,
 * scores and the weighted sum of V in the rotated domain, the output sign-undone), and
 * the hybrid layout (K stored raw, V TQ-coded); "gemma4/model.rs": the cache buffers
 * (codes [nkv, capacity, hd * bits / 8], f32 norms [nkv, capacity, hd / 256]).
 * The pages name but do not print the codebooks and sign tables: the codebook here is
 * the Lloyd-Max quantiser of the standard normal computed from its definition, and the
 * signs are an input.
 *
 * Readings (the pages leave these open): the block is min(hd, 256) dims; the norm is the
 * RMS of the rotated block (the post-scale element RMS is then the scale factor 1, the
 * "bare" setting the pages keep); an element is coded with the nearest centroid, a value
 * on a cell boundary taking the upper cell; 4-bit codes put element 2j in the low nibble
 * of byte j and element 2j+1 in the high nibble.
 */
#ifndef TQ_ORACLE_H
#define TQ_ORACLE_H
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Lloyd-Max quantiser of N(0, 1) with `levels` output levels: centroids[levels]
 * ascending, boundaries[levels + 1] with boundaries[0] = -inf and boundaries[levels] =
 * +inf.  Alternates the two optimality conditions (each boundary the midpoint of its
 * centroids, each centroid the mean of N(0,1) on its cell) until no value moves by more
 * than 1e-13; returns the number of rounds.  The levels are kept symmetric (the upper
 * half computed, the lower half its mirror), so the middle boundary is exactly 0. */
int orc_lloyd_max_normal(int levels, double* centroids, double* boundaries);
/* mean squared error E[(X - Q(X))^2] of that quantiser, X ~ N(0, 1), in closed form */
double orc_lloyd_max_mse(int levels, const double* centroids, const double* boundaries);

/* normalised Walsh-Hadamard transform (Sylvester order) of n = 2^k values, in place:
 * x <- H x / sqrt(n), H[i][j] = (-1)^popcount(i & j).  Its own inverse. */
void orc_fwht(double* x, int n);

/* rotation of one head row of hd values, block by block (blocks of min(hd, 256)):
 * x <- H (s . x) / sqrt(B); and its inverse x <- s . (H x / sqrt(B)) */
void orc_tq_rotate(double* x, int hd, const int8_t* signs);
void orc_tq_unrotate(double* x, int hd, const int8_t* signs);

/* bytes of one row's codes (hd / 2 at 4 bits, hd at 5, 6 and 8 bits), and norms per row */
int orc_tq_code_bytes(int hd, int bits);
int orc_tq_blocks(int hd);

/* encode one head row x [hd] (the appended K or V row) with `bits` in {4, 5, 6, 8}: rotate,
 * norm = sqrt(mean of the rotated block's squares), code of each element = the cell of
 * u / norm (0 when norm is 0); codes [orc_tq_code_bytes], norms [orc_tq_blocks] (f32). */
void orc_tq_encode_row(const double* x, int hd, const int8_t* signs, int bits,
                       const double* boundaries, uint8_t* codes, float* norms);
/* decode one row into the rotated domain: u_i = centroid[code_i] * norm of its block */
void orc_tq_decode_row(const uint8_t* codes, const float* norms, int hd, int bits,
                       const double* centroids, double* u);

/* attention of one query over explicit rows of a TQ cache: the query rotated, each
 * score s_j = scale * (q_rot . k_j) against the decoded (rotated) key -- or, for the
 * hybrid layout (k_codes NULL), scale * (q . K_j) against raw bf16 keys k_bf16 --,
 * optional softcap, softmax, o_rot = sum_j p_j v_j over the decoded values, o =
 * unrotate(o_rot).  Row r of a code array starts at r * code_bytes, of a norm array at
 * r * blocks, of k_bf16 at r * hd. */
void orc_attend_tq(const double* q, int hd, int bits, const int8_t* signs,
                   const double* centroids, const uint8_t* k_codes, const float* k_norms,
                   const uint16_t* k_bf16, const uint8_t* v_codes, const float* v_norms,
                   const long* rows, long n, double scale, double softcap, double* o);

#ifdef __cplusplus
}
#endif
#endif
