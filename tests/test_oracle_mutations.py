"""Planted mistakes in the oracle must trip a pin.

Each case below edits one line of a copy of oracle.cpp (a dropped term, a wrong sign,
a transposed operand or index, an off-by-one), builds the copy with the same flags as
the real oracle, and checks that at least one pin of tests/pins.py fails on it. The
real oracle passes every pin (test_oracle_pins.py), so the pins are shown to tell a
correct oracle from a plausibly broken one. Runs on the CPU only.
"""
from __future__ import annotations

import concurrent.futures as cf
import os
import tempfile

import pytest

import oracle
from tests import pins

SRC = os.path.join(os.path.dirname(oracle.__file__), "oracle.cpp")

MUTATIONS = [
    ("lu_tie_rule_last_max", "      if (v > best) {", "      if (v >= best) {"),
    ("lu_nan_candidate_wins", "      if (v > best) {", "      if (!(v <= best)) {"),
    ("lu_nan_in_place_skipped",
     "    T best = std::fabs(a(k, k));\n    for (int i = k + 1; i < n; ++i) {",
     "    T best = T(-1);\n    for (int i = k; i < n; ++i) {"),
    ("lu_search_skips_last_row",
     "    for (int i = k + 1; i < n; ++i) {\n      T v = std::fabs(a(i, k));\n      if (v > best)",
     "    for (int i = k + 1; i < n - 1; ++i) {\n      T v = std::fabs(a(i, k));\n      if (v > best)"),
    ("lu_rhs_not_swapped",
     "        T t = b(k, c);\n        b(k, c) = b(p, c);\n        b(p, c) = t;\n      }\n    }\n    const T r",
     "      }\n    }\n    const T r"),
    ("lu_L_part_not_swapped",
     "      for (int c = 0; c < n; ++c) {\n        T t = a(k, c);",
     "      for (int c = k; c < n; ++c) {\n        T t = a(k, c);"),
    ("lu_schur_sign", "a(i, j) = std::fma(-l, a(k, j), a(i, j));",
     "a(i, j) = std::fma(l, a(k, j), a(i, j));"),
    ("lu_schur_transposed_operand", "a(i, j) = std::fma(-l, a(k, j), a(i, j));",
     "a(i, j) = std::fma(-l, a(j, k), a(i, j));"),
    ("lu_forward_solve_dropped",
     "      for (int c = 0; c < nrhs; ++c) b(i, c) = std::fma(-l, b(k, c), b(i, c));\n    }\n  }\n  if (msc",
     "    }\n  }\n  if (msc"),
    ("lu_back_subst_transposed",
     "b(i, c) = std::fma(-a(i, k), x, b(i, c));\n    }\n  }\n  if (tie_step) *tie_step = tie;",
     "b(i, c) = std::fma(-a(k, i), x, b(i, c));\n    }\n  }\n  if (tie_step) *tie_step = tie;"),
    ("lu_floor_is_zero", "const bool ok = mag >= floor_v;", "const bool ok = mag > T(0);"),
    ("lu_info_off_by_one", "if (!ok && inf == 0) inf = k + 1;", "if (!ok && inf == 0) inf = k;"),
    ("lu_info_last_not_first", "if (!ok && inf == 0) inf = k + 1;", "if (!ok) inf = k + 1;"),
    ("lu_failed_x_not_zeroed",
     "    for (int i = 0; i < n * nrhs; ++i) B[i] = T(0);\n  }\n  *info = inf;",
     "  }\n  *info = inf;"),
    ("chol_sqrt_dropped", "const T l = std::sqrt(d);\n    a(k, k) = l;",
     "const T l = d;\n    a(k, k) = l;"),
    ("chol_update_writes_upper",
     "for (int i = j; i < n; ++i) a(i, j) = std::fma(-a(i, k), ljk, a(i, j));",
     "for (int i = j; i < n; ++i) a(j, i) = std::fma(-a(i, k), ljk, a(j, i));"),
    ("chol_back_solve_not_transposed",
     "b(i, c) = std::fma(-a(k, i), x, b(i, c));\n    }\n  }\n  *info = 0;",
     "b(i, c) = std::fma(-a(i, k), x, b(i, c));\n    }\n  }\n  *info = 0;"),
    ("chol_info_off_by_one", "      inf = k + 1;\n      break;", "      inf = k;\n      break;"),
    ("chol_zero_pivot_accepted", "if (!(d > T(0))) {\n      inf = k + 1;",
     "if (!(d >= T(0))) {\n      inf = k + 1;"),
    ("bdsv_trsm_uses_F_not_FT", "s = std::fma(-E[ar * bs + m], blk(k - 1, MAIN, j, m), s);",
     "s = std::fma(-E[ar * bs + m], blk(k - 1, MAIN, m, j), s);"),
    ("bdsv_syrk_transposed", "s = std::fma(-E[i * bs + m], E[j * bs + m], s);",
     "s = std::fma(-E[i * bs + m], E[m * bs + j], s);"),
    ("bdsv_forward_coupling_dropped",
     "z[i] = std::fma(-blk(k, LEFT, i, m), x[(k - 1) * bs + m], z[i]);", ";"),
    ("bdsv_backward_uses_E_not_ET",
     "z[m] = std::fma(-blk(k + 1, LEFT, i, m), x[(k + 1) * bs + i], z[m]);",
     "z[m] = std::fma(-blk(k + 1, LEFT, m, i), x[(k + 1) * bs + i], z[m]);"),
    ("bdsv_backward_trsv_not_transposed",
     "s = std::fma(-blk(k, MAIN, m, j), x[k * bs + m], s);",
     "s = std::fma(-blk(k, MAIN, j, m), x[k * bs + m], s);"),
    ("bdsv_info_local_index", "inf = k * bs + c + 1;", "inf = c + 1;"),
    ("getrs_swaps_skipped", "    if (p != k && p >= 0 && p < n)\n      for (int c = 0; c < nrhs; ++c) {",
     "    if (false)\n      for (int c = 0; c < nrhs; ++c) {"),
    ("getrs_last_row_never_swapped",
     "    if (p != k && p >= 0 && p < n)\n      for (int c = 0; c < nrhs; ++c) {",
     "    if (p != k && p >= 0 && p < n - 1)\n      for (int c = 0; c < nrhs; ++c) {"),
    ("getrs_swaps_reverse_order",
     "  for (int k = 0; k < n; ++k) {\n    const int p = ipiv[k] - 1;",
     "  for (int k = n - 1; k >= 0; --k) {\n    const int p = ipiv[k] - 1;"),
    ("getrs_forward_transposed",
     "      const T l = a(i, k);\n      for (int c = 0; c < nrhs; ++c) b(i, c) = std::fma(-l, b(k, c), b(i, c));\n    }\n  for",
     "      const T l = a(k, i);\n      for (int c = 0; c < nrhs; ++c) b(i, c) = std::fma(-l, b(k, c), b(i, c));\n    }\n  for"),
    ("getrs_back_subst_transposed",
     "b(i, c) = std::fma(-a(i, k), x, b(i, c));\n    }\n  }\n}",
     "b(i, c) = std::fma(-a(k, i), x, b(i, c));\n    }\n  }\n}"),
    ("potrs_forward_unscaled",
     "B[at(b_layout, n, nrhs, r, c)]; };\n  for (int c = 0; c < nrhs; ++c) {\n    for (int k = 0; k < n; ++k) {\n      const T y = b(k, c) * (T(1) / a(k, k));",
     "B[at(b_layout, n, nrhs, r, c)]; };\n  for (int c = 0; c < nrhs; ++c) {\n    for (int k = 0; k < n; ++k) {\n      const T y = b(k, c);"),
    ("potrs_back_solve_not_transposed",
     "b(i, c) = std::fma(-a(k, i), x, b(i, c));\n    }\n  }\n}",
     "b(i, c) = std::fma(-a(i, k), x, b(i, c));\n    }\n  }\n}"),
    ("chol_upper_fill_reads_lower",
     "  const int a_layout = fill == 0 ? layout : 1 - layout;\n  for_systems(batch, nthreads, [&](int64_t s) {\n    potrf_potrs_one<T>(a_layout, layout, n, nrhs,",
     "  const int a_layout = layout;\n  for_systems(batch, nthreads, [&](int64_t s) {\n    potrf_potrs_one<T>(a_layout, layout, n, nrhs,"),
    ("chol_upper_fill_b_transposed",
     "    potrf_potrs_one<T>(a_layout, layout, n, nrhs, A + s * n * n,",
     "    potrf_potrs_one<T>(a_layout, a_layout, n, nrhs, A + s * n * n,"),
    ("threshold_comparison_flipped", "if (akk >= bar) p = k;   // the row in place is kept",
     "if (akk <= bar) p = k;   // the row in place is kept"),
    ("threshold_pivot_magnitude_of_max", "const T mag = (p == k) ? akk : best;",
     "const T mag = best;"),
    ("ruda_pivots_not_minus_one", "    for (int k = 0; k < n; ++k) ipiv[k] = -1;\n", ""),
    ("ruda_overflow_not_reported", "    inf = -3;\n  if (inf != 0) {\n    if (ruda) {",
     "    inf = 0;\n  if (inf != 0) {\n    if (ruda) {"),
    ("ruda_symmetry_check_trivial", "        if (!(a(r, c) == a(c, r))) {",
     "        if (!(a(r, c) == a(r, c))) {"),
    ("ruda_chol_input_check_skips_b",
     "    if (!(all_finite(A, (int64_t)n * n) && all_finite(B, (int64_t)n * nrhs))) {\n      fail_ruda(-1);\n      return;\n    }\n    for (int r = 0;",
     "    if (!(all_finite(A, (int64_t)n * n))) {\n      fail_ruda(-1);\n      return;\n    }\n    for (int r = 0;"),
    ("mirror_forward_not_transposed",
     "for (int j = k + 1; j < n; ++j) b(j, c) = std::fma(-s_(k, j), z, b(j, c));",
     "for (int j = k + 1; j < n; ++j) b(j, c) = std::fma(-s_(j, k), z, b(j, c));"),
    ("mirror_swaps_in_step_order",
     "  for (int k = n - 1; k >= 0; --k) {  // x = P^T w",
     "  for (int k = 0; k < n; ++k) {  // x = P^T w"),
    ("mirror_swaps_skipped", "    if (q == k || q < 0 || q >= n) continue;", "    continue;"),
    ("mirror_backward_scaled",
     "      for (int i = 0; i < k; ++i) b(i, c) = std::fma(-s_(k, i), b(k, c), b(i, c));",
     "      for (int i = 0; i < k; ++i) b(i, c) = std::fma(-s_(k, i), b(k, c) / s_(k, k), b(i, c));"),
    ("mirror_reads_row_major", "  auto s_ = [&](int r, int c) -> T { return S[at(1, n, n, r, c)]; };",
     "  auto s_ = [&](int r, int c) -> T { return S[at(0, n, n, r, c)]; };"),
    ("il_block_offset_missing_w", "T* base(int64_t s) const { return p + (s / w) * w * size + s % w; }",
     "T* base(int64_t s) const { return p + (s / w) * size + s % w; }"),
    ("il_gather_contiguous", "for (int64_t e = 0; e < size; ++e) dst[e] = b[e * w];",
     "for (int64_t e = 0; e < size; ++e) dst[e] = b[e];"),
    ("il_ipiv_not_interleaved",
     "                          tie_step ? tie_step + s : nullptr, t, ruda, scale);\n    a.scatter(s, as.data());\n    b.scatter(s, bs.data());\n    pv.scatter(s, ps.data());",
     "                          tie_step ? tie_step + s : nullptr, t, ruda, scale);\n    a.scatter(s, as.data());\n    b.scatter(s, bs.data());\n    for (int k = 0; k < n; ++k) ipiv[s * n + k] = ps[k];"),
    ("getrf_il_ipiv_not_interleaved",
     "                       tie_step ? tie_step + s : nullptr);\n    a.scatter(s, as.data());\n    pv.scatter(s, ps.data());",
     "                       tie_step ? tie_step + s : nullptr);\n    a.scatter(s, as.data());\n    for (int k = 0; k < n; ++k) ipiv[s * n + k] = ps[k];"),
    ("mirror_il_ipiv_not_interleaved",
     "                  tie_step ? tie_step + s : nullptr, t, scale);\n    a.scatter(s, as.data());\n    b.scatter(s, bs.data());\n    pv.scatter(s, ps.data());",
     "                  tie_step ? tie_step + s : nullptr, t, scale);\n    a.scatter(s, as.data());\n    b.scatter(s, bs.data());\n    for (int k = 0; k < n; ++k) ipiv[s * n + k] = ps[k];"),
    ("il_chol_fill_ignored",
     "    potrf_potrs_ex_one<T>(a_layout, layout, n, nrhs, as.data(), bs.data(), info + s, ruda);",
     "    potrf_potrs_ex_one<T>(layout, layout, n, nrhs, as.data(), bs.data(), info + s, ruda);"),
    ("il_threshold_dropped",
     "                          tie_step ? tie_step + s : nullptr, t, ruda, scale);",
     "                          tie_step ? tie_step + s : nullptr, T(1), ruda, scale);"),
    ("il_chol_contract_dropped",
     "    potrf_potrs_ex_one<T>(a_layout, layout, n, nrhs, as.data(), bs.data(), info + s, ruda);",
     "    potrf_potrs_ex_one<T>(a_layout, layout, n, nrhs, as.data(), bs.data(), info + s, 0);"),
    ("mirror_scaling_dropped",
     "  getrf_getrs_ex_one<T>(1, n, 0, As, nullptr, ipiv, inf, tie, t, 0, scale);",
     "  getrf_getrs_ex_one<T>(1, n, 0, As, nullptr, ipiv, inf, tie, t, 0, 0);"),
    ("mirror_failed_x_not_zeroed",
     "  getrs_mirror_one<T>(layout, n, nrhs, As, ipiv, Bs);\n  if (*inf != 0)\n    for (int i = 0; i < n * nrhs; ++i) Bs[i] = T(0);",
     "  getrs_mirror_one<T>(layout, n, nrhs, As, ipiv, Bs);"),
    ("getrs_il_pivots_not_gathered", "    pv.gather(s, ps.data());",
     "    for (int k = 0; k < n; ++k) ps[k] = ipiv[s * n + k];"),
    ("potrf_il_fill_ignored",
     "    potrf_potrs_one<T>(a_layout, layout, n, 0, as.data(), nullptr, info + s);",
     "    potrf_potrs_one<T>(layout, layout, n, 0, as.data(), nullptr, info + s);"),
    ("potrs_il_fill_ignored",
     "    potrs_one<T>(a_layout, layout, n, nrhs, as.data(), bs.data());",
     "    potrs_one<T>(layout, layout, n, nrhs, as.data(), bs.data());"),
    ("scaling_u_not_restored", "      for (int j = k; j < n; ++j) a(k, j) = a(k, j) * msc;   // U's scale restored",
     "      for (int j = k; j < n; ++j) a(k, j) = a(k, j);   // U's scale restored"),
    ("scaling_restores_l_too", "      for (int j = k; j < n; ++j) a(k, j) = a(k, j) * msc;   // U's scale restored",
     "      for (int j = 0; j < n; ++j) a(k, j) = a(k, j) * msc;   // U's scale restored"),
    ("scaling_first_row_max", "    for (int i = 0; i < n * n; ++i)\n      if (std::fabs(A[i]) > msc) msc = std::fabs(A[i]);",
     "    for (int i = 0; i < n; ++i)\n      if (std::fabs(A[i]) > msc) msc = std::fabs(A[i]);"),
    ("scaling_multiplies", "      for (int i = 0; i < n * n; ++i) A[i] = A[i] / msc;",
     "      for (int i = 0; i < n * n; ++i) A[i] = A[i] * msc;"),
    ("bdmv_window_one_block_late", "const T* xw = xpad + (int64_t)br * bs;",
     "const T* xw = xpad + (int64_t)(br + 1) * bs;"),
    ("bdmv_output_into_pad", "ypad[(int64_t)(br + 1) * bs + row] = acc;",
     "ypad[(int64_t)br * bs + row] = acc;"),
    ("bdmv_right_block_dropped", "for (int c = 0; c < w; ++c) acc = std::fma(srow[c], xw[c], acc);",
     "for (int c = 0; c < 2 * bs; ++c) acc = std::fma(srow[c], xw[c], acc);"),
    ("bdmv_blocks_transposed", "acc = std::fma(srow[c], xw[c], acc);",
     "acc = std::fma(strips[strip_at(bs, br, c / bs, c % bs, row)], xw[c], acc);"),
]


def _build_variant(tmpdir, name, old, new):
    src = open(SRC).read()
    assert src.count(old) == 1, f"mutation {name}: pattern must occur exactly once"
    path = os.path.join(tmpdir, f"{name}.cpp")
    with open(path, "w") as f:
        f.write(src.replace(old, new))
    return oracle.compile_library(path, os.path.join(tmpdir, f"lib{name}.so"))


@pytest.fixture(scope="module")
def variants():
    with tempfile.TemporaryDirectory() as d:
        with cf.ThreadPoolExecutor(max_workers=min(8, os.cpu_count() or 1)) as ex:
            futs = {m[0]: ex.submit(_build_variant, d, *m) for m in MUTATIONS}
            libs = {k: f.result() for k, f in futs.items()}
        yield libs


@pytest.mark.parametrize("name", [m[0] for m in MUTATIONS])
def test_planted_mistake_trips_a_pin(variants, name):
    orc = oracle.Oracle(variants[name])
    assert pins.failing_pins(orc), f"no pin caught the planted mistake {name}"
