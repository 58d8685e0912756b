"""Writes hand_worked_cases.json: decode cases whose answers follow in closed
form from the definition of decode attention (each case's "derivation" says
how), computed here with the logistic function -- no oracle, no GPU.

    python tests/golden/make_hand_worked_cases.py

tests/test_oracle_pins.py checks that the stored file equals what this script
builds, and pins the oracle against it.
"""
import json
import math
import os

HERE = os.path.dirname(os.path.abspath(__file__))
PATH = os.path.join(HERE, "hand_worked_cases.json")

ABOUT = (
    "Hand-worked decode cases whose answers follow in closed form from the definition of "
    "decode attention: out[b,h] = softmax(scale * q[b,h] . K^T) . V over the tokens reached "
    "through the block table. Sources: 'benchmark_decoding.py' (function reference_output: the "
    "float32 definition; setup_test_data: tensor layouts), MiniVLLM docs 'Decoding Benchmark' "
    "(section 'Block table lookup mechanics': token t lives in block block_tables[b][t // "
    "block_size] at slot t % block_size, -1 = unallocated), and the Triton (new) kernel on the "
    "same page (kv head = h // (num_heads / num_kv_heads); -1 entries are masked out of the "
    "softmax). With two attended tokens whose scores differ by x, the softmax weights are the "
    "logistic values sigma(x) = 1/(1+exp(-x)) and 1 - sigma(x); with one-hot value rows the "
    "output is exactly those weights. Layouts: q [B][H][D]; caches [num_blocks][block_size]"
    "[num_kv_heads][D]; tables [B][max_blocks]. All inputs are exactly representable in fp16.")


def sigma(x):
    return 1.0 / (1.0 + math.exp(-x))


def cases():
    shuffled = dict(q=[[[1, 0]]], k_cache=[[[[0, 0]]], [[[5, 5]]], [[[1, 0]]]],
                    v_cache=[[[[0, 1]]], [[[7, 7]]], [[[1, 0]]]], block_tables=[[2, 0]],
                    context_lens=[2])
    return [
        dict(name="two_tokens_shuffled_blocks_scale1",
             derivation="token 0 sits in block 2, token 1 in block 0 (block 1 is never referenced "
                        "and holds decoy values). s = scale*(q.K0, q.K1) = (1, 0); weights = "
                        "(sigma(1), sigma(-1)); V0 = (1,0), V1 = (0,1) so out = (sigma(1), "
                        "sigma(-1)).",
             scale=1.0, **shuffled, expected=[[[sigma(1), sigma(-1)]]]),
        dict(name="two_tokens_shuffled_blocks_scale_half",
             derivation="as above with scale = 0.5: s = (0.5, 0); out = (sigma(0.5), sigma(-0.5)). "
                        "A dropped scale gives sigma(1) instead.",
             scale=0.5, **shuffled, expected=[[[sigma(0.5), sigma(-0.5)]]]),
        dict(name="gqa_head_map",
             derivation="4 query heads share 2 kv heads (group 2): heads 0,1 read kv head 0, heads "
                        "2,3 read kv head 1. Both tokens sit in block 0 (slots 0 and 1). kv head 0 "
                        "scores (1, 0); kv head 1 scores (0, 1); V rows are one-hot (1,0) then "
                        "(0,1) for both kv heads. So heads 0,1 give (sigma(1), sigma(-1)) and heads "
                        "2,3 give (sigma(-1), sigma(1)). Mapping h -> h % num_kv_heads instead "
                        "would swap heads 1 and 2.",
             scale=1.0, q=[[[1, 0], [1, 0], [1, 0], [1, 0]]],
             k_cache=[[[[1, 0], [0, 0]], [[0, 0], [1, 0]]]],
             v_cache=[[[[1, 0], [1, 0]], [[0, 1], [0, 1]]]], block_tables=[[0]],
             context_lens=[2],
             expected=[[[sigma(1), sigma(-1)], [sigma(1), sigma(-1)], [sigma(-1), sigma(1)],
                        [sigma(-1), sigma(1)]]]),
        dict(name="masked_table_entry",
             derivation="block_size 1; the table row (0, -1, 1) leaves token 1 unallocated, so "
                        "only tokens 0 and 2 are attended: s = (1, 0), out = (sigma(1), "
                        "sigma(-1)). Reading -1 as the last block (Python wrap-around) would "
                        "attend block 1 twice and give (e/(e+2), 2/(e+2)) = (0.5761, 0.4239).",
             scale=1.0, q=[[[1, 0]]], k_cache=[[[[1, 0]]], [[[0, 0]]]],
             v_cache=[[[[1, 0]]], [[[0, 1]]]], block_tables=[[0, -1, 1]], context_lens=[3],
             expected=[[[sigma(1), sigma(-1)]]]),
        dict(name="empty_context",
             derivation="context length 0: no token is attended; the pages' formula is 0/0, read "
                        "here as an all-zero output row.",
             scale=1.0, q=[[[1, 0]]], k_cache=[[[[1, 0]]]], v_cache=[[[[3, 4]]]],
             block_tables=[[0]], context_lens=[0], expected=[[[0.0, 0.0]]]),
    ]


def build():
    return {"about": ABOUT, "cases": cases()}


if __name__ == "__main__":
    with open(PATH, "w") as f:
        json.dump(build(), f, indent=2)
        f.write("\n")
    print("wrote", PATH)
