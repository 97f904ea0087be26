"""Admission arithmetic of the capacity comparison (host logic, no GPU).

At a fixed one-layer KV budget, admission_cap gives the pages in the pool,
the pages one request needs and the requests admitted.  It is checked
against admitting requests one at a time until the free pages run out, and
against the pages' own claim that the e4m3 cache holds twice the tokens of
the BF16 one in the same memory ("Cosa ha cambiato Cloudflare per Kimi e GLM":
about 686 k against 1.37 M tokens)."""
import pytest

from fp8_paged_kv_gb300.pool import admission_cap


def _admit_one_by_one(budget, context, Hkv, D, ps, elem_bytes):
    page_bytes = 0
    for _ in range(2):          # K and V
        page_bytes += Hkv * ps * D * elem_bytes
    free = 0
    while (free + 1) * page_bytes <= budget:
        free += 1
    need = 0
    while need * ps < context:
        need += 1
    n = 0
    while need and free >= need:
        free -= need
        n += 1
    return n


@pytest.mark.parametrize("fp8", [True, False])
@pytest.mark.parametrize("budget_gib,context,Hkv,ps", [(4, 8192, 8, 16), (4, 8193, 8, 16), (1, 131072, 8, 64),
                                                      (0.5, 1000, 2, 32), (4, 8192, 1, 256)])
def test_cap_matches_one_by_one_admission(fp8, budget_gib, context, Hkv, ps):
    budget = int(budget_gib * 2**30)
    pages, per_req, cap = admission_cap(budget, context, Hkv=Hkv, D=128, page_size=ps, fp8=fp8)
    assert per_req == -(-context // ps)
    assert pages * 2 * Hkv * ps * 128 * (1 if fp8 else 2) <= budget
    assert cap == _admit_one_by_one(budget, context, Hkv, 128, ps, 1 if fp8 else 2)


def test_e4m3_doubles_the_tokens_of_bf16_at_the_headline_shape():
    budget = 4 * 2**30
    _, _, bf16 = admission_cap(budget, 8192, Hkv=8, D=128, page_size=16, fp8=False)
    _, _, fp8 = admission_cap(budget, 8192, Hkv=8, D=128, page_size=16, fp8=True)
    assert (bf16, fp8) == (128, 256)
    assert fp8 * 8192 == 2 * bf16 * 8192


def test_nothing_fits_in_less_than_one_request():
    pages, per_req, cap = admission_cap(1 << 20, 8192, Hkv=8, D=128, page_size=16, fp8=True)
    assert pages == 32 and per_req == 512 and cap == 0
    assert admission_cap(1 << 20, 0, Hkv=8, D=128, page_size=16, fp8=True)[2] == 0
