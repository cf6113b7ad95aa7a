"""Plant plausible mistakes in copies of the CPU oracle and require the pins to
catch each one.  Mutants are compiled from text-edited copies of
oracle/msa_ref.c into a temporary directory; the committed oracle is untouched.
"""
import os
import shutil
import subprocess

import numpy as np
import pytest

import oracle
from tests import test_oracle as pins
from tests import test_oracle_kl as klpins
from tests import test_oracle_quality as qpins

SRC = os.path.join(os.path.dirname(oracle.__file__), "msa_ref.c")

MUTANTS = {
    # tie rule reversed: equal pooled scores rank the higher block id first
    "tie_reversed": ("return (x->blk > y->blk) - (x->blk < y->blk);",
                     "return (x->blk < y->blk) - (x->blk > y->blk);"),
    # min pooling instead of max pooling
    "min_pool": ("if (s > best) best = s;", "if (best == -INFINITY || s < best) best = s;"),
    # sum pooling instead of max pooling
    "sum_pool": ("if (s > best) best = s;", "best = (best == -INFINITY ? 0.0 : best) + s;"),
    # plain top-16 of the candidates: the local block is not forced in
    "local_not_forced": ("\n    s[0] = (int32_t)lb;",
                         "\n    s[0] = lb >= p->topk ? cand[p->topk - 1].blk : (int32_t)lb;"),
    # causal clip of the local block dropped
    "no_causal_clip": ("if (tok > t) continue;\n          krow[n]", "(void)0;\n          krow[n]"),
    # softmax scale dropped
    "no_scale": ("z[i] = s * p->scale;\n      }\n      softmax_combine",
                 "z[i] = s;\n      }\n      softmax_combine"),
    # wrong KV head for a query head (reversed group order)
    "wrong_kv_head": ("krow[n] = k + (size_t)tok * row + (size_t)g * p->D;\n          vrow",
                      "krow[n] = k + (size_t)tok * row + (size_t)(p->G - 1 - g) * p->D;\n          vrow"),
    # index dot product over one dimension too few
    "dropped_index_term": ("for (int d = 0; d < p->Di; ++d) s += bf16_to_double(qg[d])",
                           "for (int d = 1; d < p->Di; ++d) s += bf16_to_double(qg[d])"),
    # softmax normaliser off by one
    "bad_normaliser": ("for (int d = 0; d < D; ++d) out[d] /= l;",
                       "for (int d = 0; d < D; ++d) out[d] /= (l + 1.0);"),
    # selection quality: block masses not normalised by the softmax sum
    "quality_unnormalised_mass": ("Ah[i / p->block] += z[i] / Z;", "Ah[i / p->block] += z[i];"),
    # selection quality: ideal selection ranked by the group's last head only
    "quality_last_head_only": ("P[b] += Ah[b] / hpg;", "P[b] = Ah[b];"),
    # selection quality: local block not forced into the ideal selection
    "quality_local_not_forced": ("ds[0] = (int32_t)lb;",
                                 "ds[0] = lb >= p->topk ? cand[p->topk - 1].blk : (int32_t)lb;"),
    # selection quality: every head scored with its group's first head
    "quality_wrong_head": ("const uint16_t *qh = q_t + (size_t)(g * hpg + hh) * p->D;\n      /*",
                           "const uint16_t *qh = q_t + (size_t)(g * hpg) * p->D;\n      /*"),
    # selection quality: softmax scale dropped
    "quality_no_scale": ("z[i] = s * p->scale;\n        if (z[i] > m)",
                         "z[i] = s;\n        if (z[i] > m)"),
    # KL: the divergence taken the other way round, D_KL(Q || P)
    "kl_reversed": ("if (P[j] > 0.0) loss += P[j] * (log(P[j]) - log(Q[j]));",
                    "loss += Q[j] * (log(Q[j]) - log(P[j]));"),
    # KL: gradient of the pooled scores with the wrong sign
    "kl_grad_sign": ("const double dz = Q[j] - P[j];", "const double dz = P[j] - Q[j];"),
    # KL: teacher not averaged over the group's heads
    "kl_heads_summed": ("P[j] += exp(z[i++] - m) / Z / hpg;", "P[j] += exp(z[i++] - m) / Z;"),
    # KL: a tied pooled maximum credited to the last token
    "kl_tie_last": ("if (s > zi[j]) { /* strictly", "if (s >= zi[j]) { /* strictly"),
    # KL: pooled index scores of the local block include tokens after t
    "kl_pool_not_causal": ("        if (tok > t) continue;\n        const uint16_t *kr = k_idx",
                           "        const uint16_t *kr = k_idx"),
    # selection quality: the full softmax stops at the local block's start
    "quality_no_local_tokens": ("      for (int64_t i = 0; i <= t; ++i) {\n        const uint16_t *kr",
                                "      for (int64_t i = 0; i < lb * p->block; ++i) {\n        const uint16_t *kr"),
}

PINS = [
    lambda r: pins.test_selection_equals_bruteforce_small_blocks(r, 4, 5, 3, 2),
    lambda r: pins.test_selection_equals_bruteforce_small_blocks(r, 8, 6, 4, 8),
    pins.test_selection_equals_bruteforce_block128,
    pins.test_needle_block_is_selected,
    pins.test_short_context_equals_full_causal_attention,
    pins.test_sparse_equals_masked_sdpa,
    pins.test_closed_forms,
    qpins.test_quality_block_masses_and_ideal_selection_match_sdpa,
    qpins.test_quality_short_context_recalls_everything,
    qpins.test_quality_dominant_key_closed_form,
    qpins.test_quality_ideal_selection_dominates_the_index_selection,
    klpins.test_single_candidate_gives_zero_loss_and_gradient,
    klpins.test_teacher_and_student_distributions,
    klpins.test_gradients_match_finite_differences_of_the_loss,
    klpins.test_tied_maximum_sends_the_gradient_to_the_first_token,
]


@pytest.fixture(scope="module")
def mutant_dir(tmp_path_factory):
    return tmp_path_factory.mktemp("mutants")


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_pins_catch_mutant(name, mutant_dir):
    old, new = MUTANTS[name]
    text = open(SRC).read()
    assert text.count(old) == 1, "mutation site must exist exactly once"
    d = mutant_dir / name
    d.mkdir()
    shutil.copy(os.path.join(os.path.dirname(SRC), "msa_ref.h"), d / "msa_ref.h")
    (d / "msa_ref.c").write_text(text.replace(old, new))
    so = str(d / "libmut.so")
    subprocess.check_call(["gcc", "-O2", "-std=c99", "-fopenmp", "-fPIC", "-shared",
                           str(d / "msa_ref.c"), "-o", so, "-lm"])
    caught = []
    with oracle.use_library(so):
        for pin in PINS:
            try:
                pin(oracle)
            except (AssertionError, ValueError):
                caught.append(pin)
    assert caught, "mutant %s passed every pin" % name
