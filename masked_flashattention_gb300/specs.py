"""MaskSpecs of the five workloads, forward and backward.

A MaskSpec groups descriptor rows into Regions, each with a row guard and a visibility rule
(CompileMask section 3.2.1).  In a forward spec the row index i is a query row and j a key; in a
backward spec i is a key column and j a query row: the paper builds the backward descriptor
from its own MaskSpec so that its intervals follow the backward traversal (section 3.2.2 / 3.3).

Segment conventions (metadata, see ``workloads``):
  1  documents; 2  one segment; 3  segment 0 = prompt, then responses;
  4  segment 0 = history, segment 1 = candidates; 5  segment 0 = system prefix, then documents;
  6  users packed back to back, user u = history segment 2u and candidate segment 2u + 1.
"""

FWD = {
    1: """
# packed documents: row i sees its own document up to itself
region all : j >= seg_start(i) && j <= i
""",
    2: """
# causal
region all : j <= i
""",
    3: """
# shared-prompt reward model: prompt rows are causal; a response row sees the prompt and its
# own response up to itself (the two-slot Region of the paper's worked example)
region seg_idx(i) == 0 : j <= i
region seg_idx(i) >= 1 : j < seg_end_at(0) || (j >= seg_start(i) && j <= i)
""",
    4: """
# HSTU: history rows are causal; a candidate sees the history and itself
region seg_idx(i) == 0 : j <= i
region seg_idx(i) >= 1 : j < seg_end_at(0) || j == i
""",
    5: """
# three-interval packing: prefix rows are causal; a document row sees the prefix, the first 64
# tokens of the previous document (none for the first document) and its own document causally
region seg_idx(i) == 0 : j <= i
region seg_idx(i) >= 1 : j < seg_end_at(0) || (seg_idx(i) >= 2 && j >= seg_start_at(seg_idx(i) - 1) && j < min(seg_start_at(seg_idx(i) - 1) + 64, seg_end_at(seg_idx(i) - 1))) || (j >= seg_start(i) && j <= i)
""",
    6: """
# variable-length packed HSTU: per user, history rows are causal within the history; a candidate
# row sees its user's history (the previous segment) and itself
region seg_idx(i) % 2 == 0 : j >= seg_start(i) && j <= i
region seg_idx(i) % 2 == 1 : (j >= seg_start_at(seg_idx(i) - 1) && j < seg_start(i)) || j == i
""",
}

BWD = {
    1: """
# key column i is seen by the rows of its document from i on
region all : j >= i && j < seg_end(i)
""",
    2: """
region all : j >= i
""",
    3: """
# prompt keys are seen by later prompt rows and every response row; response keys by later rows
# of the same response
region seg_idx(i) == 0 : j >= i
region seg_idx(i) >= 1 : j >= i && j < seg_end(i)
""",
    4: """
# history keys are seen by later history rows and every candidate; a candidate key only by itself
region seg_idx(i) == 0 : j >= i
region seg_idx(i) >= 1 : j == i
""",
    5: """
# prefix keys are seen by later prefix rows and every document row; a document key by later rows
# of its document and, within the document's first 64 tokens, by every row of the next document
region seg_idx(i) == 0 : j >= i
region seg_idx(i) >= 1 : (j >= i && j < seg_end(i)) || (i < seg_start(i) + 64 && j >= seg_start_at(seg_idx(i) + 1) && j < seg_end_at(seg_idx(i) + 1))
""",
    6: """
# a history key is seen by the later history rows and all candidates of its user (the next
# segment); a candidate key only by itself
region seg_idx(i) % 2 == 0 : j >= i && j < seg_end_at(seg_idx(i) + 1)
region seg_idx(i) % 2 == 1 : j == i
""",
}
