"""Plain, slow, fp64 CPU oracle for the NSA / DSA forward hot path.

TEST INFRASTRUCTURE ONLY.  Nothing in the product package may import, call or
execute this package: only ``tests/``, ``__graft_entry__.smoke()`` and the
``cpu_baseline`` / ``--impl reference`` legs of ``bench.py`` use it.  It
shares no code with the CUDA path (it reads the same seeded inputs from
``workloads``, which holds no arithmetic of the method).

Sources (untrusted web pages, cited by title and section):
  [P1] "DeepSeek의 획기적인 AI 혁신: NSA, 비용 절감 및 장문맥 언어 모델 성능 강화"
       (news article): key points list, "hardware-aware design" section.
  [P2] "AI 모델의 '긴 문장 처리' 한계 돌파, 딥시크의 새 어텐션 기술 화제" (blog):
       section II (three paths, hyper-parameters l=32, d=16, l'=64,
       n=16 incl. 1 initial + 2 local blocks, w=512), section III.3
       (64k decode reads 5,632 tokens instead of 65,536).
  [P3] deepdaiv newsletter no. 82 on sparse attention: the token-compression,
       token-selection and sliding-window paragraphs.
  [P4] "딥시크 희소 어텐션 DSA 원리: 라이트닝 인덱서와 상위 2048 토큰 선택 구조 해설":
       "쉽게 이해하기" (indexer = weighted sum of ReLU dot products, keys shared
       by heads; keep the top 2048 positions; softmax over the selected set
       only; selection independent per query position) and the key-message
       list (2048 = 1.6% of 128k).

Readings taken where the pages are silent are listed in each function's
docstring.  Parity status per function:
  bf16_round ............ pinned (torch fp32->bf16 on fp32-exact inputs)
  compress .............. pinned (mean-pool closed form; torch.matmul)
  cmp_attention ......... pinned (textbook softmax attention when all blocks
                          visible; empty set gives 0)
  block_scores .......... pinned (conservation sum = (l/d)*heads; brute
                          overlap count on tiny cases)
  select_blocks ......... pinned (brute-force stable sort; forced blocks)
  sel / win attention ... pinned (n*l' >= T or w >= T reduces to full causal
                          attention by a textbook formula)
  combined output ....... pinned (an independent torch formulation of the
                          whole forward on the same kept blocks and cache;
                          out = sum of gate x branch output)
  dsa_decode ............ pinned (k >= T reduces to full softmax attention;
                          brute-force top-k; 131072/2048 = 64)
  dsa_prefill ........... pinned (topk >= t+1 reduces to textbook causal
                          attention; last row = the decode step; brute-force
                          loops and tuple sort for the kept sets)
  decode_multi .......... pinned (m = 1 is the decode step bit for bit; rows
                          equal the prefill rows of token-major copies)
  nsa_bwd (backward) .... pinned (central finite differences of the forward
                          with the selection fixed; torch autograd of an
                          independent torch forward; one-key and mean-pool
                          closed forms)
"""
from .nsa import *  # noqa: F401,F403
from .dsa import *  # noqa: F401,F403
