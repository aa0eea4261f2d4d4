"""GB300-native (sm_103a) hot path of one EAGLE-2 speculative-decoding verify
step: draft-tree build, tree-masked GQA attention, acceptance walk."""
