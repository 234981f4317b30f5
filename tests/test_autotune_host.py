"""Host logic of the chunk-size autotuner (no GPU): the candidate set."""
import torch

from paged_attention_decode_gb300 import autotune as T


def test_candidates_include_default_powers_of_two_and_wave_fits():
    # 16 requests of 2048 one-token pages, one KV head: the binary-search default for a 152-CTA target is
    # 227 pages (16 x 10 = 160 CTAs, a second wave of 8); 228 pages gives 16 x 9 = 144 CTAs in one wave
    indptr = torch.arange(0, 17 * 2048, 2048)
    c = T.candidates(indptr, 1, 1, 152, 227, 1, 2048)
    assert 227 in c and 228 in c
    assert all(p in c for p in (1, 2, 4, 8, 16, 32, 64, 128, 256, 512, 1024, 2048))
    assert c == sorted(c)


def test_wave_fit_is_the_smallest_size_within_k_waves():
    indptr = torch.tensor([0, 2048])      # one request, 8 KV heads, 152-CTA waves
    c = T.candidates(indptr, 8, 1, 152, 108, 1, 2048)
    # 1 wave: 19 chunks x 8 = 152 -> ppc 108; 2 waves: 38 chunks -> ppc 54; 3 waves: 57 chunks -> ppc 36
    assert {108, 54, 36} <= set(c)
    for ppc, waves in ((108, 1), (54, 2), (36, 3)):
        assert T._chunks([2048], ppc) * 8 <= waves * 152 < T._chunks([2048], ppc - 1) * 8


def test_sizes_below_the_default_with_its_cta_count():
    # 32768 tokens of 16-token pages, 8 KV heads: the default 113 pages makes 19 chunks; so does every
    # size down to 108 (ceil(2048 / 107) = 20), and those five are candidates -- 112 = 8 x 14 among them
    indptr = torch.tensor([0, 2048])
    c = T.candidates(indptr, 8, 1, 152, 113, 1, 2048)
    assert {108, 109, 110, 111, 112, 113} <= set(c) and 107 not in c
    for ppc in range(108, 114):
        assert T._chunks([2048], ppc) == 19
    assert T._chunks([2048], 107) == 20
    # at most `same_ctas` of them
    c3 = T.candidates(indptr, 8, 1, 152, 113, 1, 2048, same_ctas=3)
    assert {110, 111, 112} <= set(c3) and 109 not in c3
