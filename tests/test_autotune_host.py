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
